// Host check of the stream-K work split (Sched in pnq_streamk.cuh) that the tensor-core GEMV
// kernels share. Everything here runs on the CPU: for many (row tiles T, K units U, grid G,
// item order) configurations it walks the items the way the kernels do (a CTA takes its items
// in index order) and checks Sched's answers against brute force:
//   - item <-> (tile, unit) is a bijection onto [0, T) x [0, U);
//   - first / owner split the items into G contiguous shares;
//   - the reducer's shares of each tile partition its units; a tile is either written whole by
//     one share or by exactly shares(t) partial shares (the tile counter's target), whose
//     workspace slots (their first units) are the ones the finishing CTA reads;
//   - every unit of a CTA's share lies inside span(i0, i1) units from its first unit (the
//     resident operand slots).
// Prints "ok <configurations>" and exits 0, or prints the first failure and exits 1.
#include "pnq_streamk.cuh"

#include <cstdio>
#include <set>
#include <vector>

namespace {

int failures = 0;

#define CHECK(cond, ...)                                                                         \
    do {                                                                                         \
        if (!(cond)) {                                                                           \
            if (failures++ == 0) {                                                               \
                std::printf("FAIL %s:%d: %s | ", __FILE__, __LINE__, #cond);                     \
                std::printf(__VA_ARGS__);                                                        \
                std::printf("\n");                                                               \
            }                                                                                    \
            return;                                                                              \
        }                                                                                        \
    } while (0)

struct Share {
    int cta, t, u_first, n_run;
};

void check(int T, int U, int G, int tile_major, int tg) {
    pnq::Sched sc{T * U, T, U, G, tile_major, tg};
    const int items = T * U;
#define CFG "T=%d U=%d G=%d tile_major=%d tg=%d", T, U, G, tile_major, tg
    // bijection
    std::vector<int> seen(items, 0);
    for (int i = 0; i < items; ++i) {
        const int t = sc.tile_of(i), u = sc.unit_of(i);
        CHECK(t >= 0 && t < T && u >= 0 && u < U, CFG);
        CHECK(sc.item(t, u) == i, CFG);
        ++seen[t * U + u];
    }
    for (int k = 0; k < items; ++k) CHECK(seen[k] == 1, CFG);
    // contiguous shares
    CHECK(sc.first(0) == 0 && sc.first(G) == items, CFG);
    for (int c = 0; c < G; ++c) {
        CHECK(sc.first(c) <= sc.first(c + 1), CFG);
        for (int i = sc.first(c); i < sc.first(c + 1); ++i) CHECK(sc.owner(i) == c, CFG);
    }
    // the reducer's walk: a share ends where the next item's tile differs, or at the CTA's end
    std::vector<Share> shares;
    for (int c = 0; c < G; ++c) {
        const int i0 = sc.first(c), i1 = sc.first(c + 1);
        if (i1 <= i0) continue;
        const int span = sc.span(i0, i1);
        const int u0 = sc.unit_of(i0);
        CHECK(span >= 1 && span <= U, CFG);
        int u_first = sc.unit_of(i0), n_run = 0;
        for (int i = i0; i < i1; ++i) {
            const int t = sc.tile_of(i), u = sc.unit_of(i);
            CHECK(((u - u0) % U + U) % U < span, "unit outside the resident span; " CFG);
            ++n_run;
            const bool last = (i + 1 == i1) || sc.tile_of(i + 1) != t;
            if (!last) {
                CHECK(sc.unit_of(i + 1) == (u + 1) % U || sc.unit_of(i + 1) == u + 1, "run skips a unit; " CFG);
                continue;
            }
            shares.push_back(Share{c, t, u_first, n_run});
            if (i + 1 < i1) u_first = sc.unit_of(i + 1);
            n_run = 0;
        }
    }
    // per tile: units covered once; whole tile alone, or shares(t) partial shares whose slots
    // are the ones finish_tile enumerates
    for (int t = 0; t < T; ++t) {
        std::vector<int> cover(U, 0);
        int whole = 0, partial = 0;
        std::set<int> slots;
        for (const Share& s : shares) {
            if (s.t != t) continue;
            for (int k = 0; k < s.n_run; ++k) {
                const int u = s.u_first + k;
                CHECK(u < U, "share runs past the last unit; " CFG);
                ++cover[u];
            }
            if (s.n_run == U) {
                ++whole;
            } else {
                ++partial;
                slots.insert(s.u_first);
            }
        }
        for (int u = 0; u < U; ++u) CHECK(cover[u] == 1, "tile %d unit %d covered %d times; " CFG, t, u, cover[u]);
        if (whole) {
            CHECK(whole == 1 && partial == 0, CFG);
            continue;
        }
        CHECK(partial == sc.shares(t), "tile %d: %d partial shares, counter target %d; " CFG, t, partial, sc.shares(t));
        CHECK(static_cast<int>(slots.size()) == partial, "two shares of tile %d in one slot; " CFG, t);
        // finish_tile's enumeration of the slots
        const bool consec = sc.consecutive(t);
        const int a0 = sc.item(t, 0);
        const int c_lo = consec ? sc.owner(a0) : 0;
        const int n = consec ? sc.owner(a0 + U - 1) - c_lo + 1 : U;
        CHECK(n == partial, CFG);
        std::set<int> read;
        for (int j = 0; j < n; ++j) read.insert(!consec ? j : (j == 0 ? 0 : sc.first(c_lo + j) - a0));
        CHECK(read == slots, "tile %d: the finisher reads other slots than the shares wrote; " CFG, t);
    }
#undef CFG
}

}  // namespace

int main() {
    // row tiles and K units of the workload's projections (128-row tiles; K units of 8 PN blocks
    // or 256 NVFP4 weights) and small edge cases
    const int Ts[] = {1, 2, 3, 5, 8, 13, 20, 40, 68, 96, 136};
    const int Us[] = {1, 2, 3, 7, 8, 10, 12, 20, 34, 68};
    const int Gs[] = {1, 2, 3, 5, 7, 8, 13, 40, 64, 80, 96, 136, 151, 152, 300, 1000};
    int n = 0;
    for (int T : Ts)
        for (int U : Us)
            for (int G : Gs) {
                if (G > T * U) continue;
                check(T, U, G, 1, 1);
                ++n;
                for (int tg : {1, 2, 3, 4, 7, 8, 16, T}) {
                    if (tg < 1 || tg > T) continue;
                    check(T, U, G, 0, tg);
                    ++n;
                }
                if (failures) return 1;
            }
    std::printf("ok %d\n", n);
    return failures ? 1 : 0;
}
