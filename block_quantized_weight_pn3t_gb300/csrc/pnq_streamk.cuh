// pnq_streamk.cuh -- the work split shared by the tensor-core GEMV kernels (PN and NVFP4).
//
// Items are 128 weight rows x one K unit; a persistent grid takes equal contiguous shares of
// them (stream-K). Consumer warps leave each finished tile's row sums in shared memory; a reducer
// warp writes a tile the CTA covered whole straight to Y, and otherwise stores the CTA's share of
// it in a workspace slot; at the end the CTA counts its shares (one atomic each) and the CTA
// that completes a tile sums its slots in unit order (so results do not depend on timing).
//
// Operands. The x fragments an item multiplies with depend only on its K unit. When the operands
// of all units of a CTA's share fit in shared memory (resident mode), the consumer and builder
// warps build them together once, before the first item (this overlaps the first weight copies),
// and the items then run without further synchronisation. Otherwise (wide batches) builder warps
// make them for each run of consecutive items with the same unit into a ring of RB slots (full /
// empty mbarriers) ahead of the consumers, from x copied into shared memory with cp.async (XB
// buffers), so shared memory does not grow with the share.
#pragma once

#include <cstdint>

#include "pnq_device.cuh"

namespace pnq {
namespace {

constexpr int kTileRows = 128;        // rows per item
constexpr int kPartPitch = 132;       // floats per (half, buffer, m) row-sum vector in shared memory
constexpr int kMaxStages = 8;
constexpr unsigned kStaticWeights = 1u;
constexpr unsigned kResident = 2u;  // operands of the whole share built in the prologue
constexpr unsigned kXOverlap = 4u;  // ... from x held in the last weight stages until then
constexpr size_t kSmemLimit = 227u * 1024u;

// Item numbering. Tile-major (item = t * U + u): a CTA's share covers one or two row tiles and
// at most U units, and it accumulates a tile over consecutive items. Grouped unit-major: row
// tiles in groups of tg (the last may be smaller), the groups one after another, inside a group
// item = base + u * n + (t - t0) (n tiles from t0): a CTA's share touches few units (so the
// operands of wide batches fit), every item of a group of n >= 2 tiles is a share of its own,
// and the tiles complete group by group. CTA c of G takes items [c * items / G, (c+1) * items / G).
struct Sched {
    int items;  // T * U < 2^31 (checked by the host)
    int T, U, G, tile_major, tg;
    __host__ __device__ int group_items() const { return tg * U; }
    __host__ __device__ int tile_of(int i) const {
        if (tile_major) return i / U;
        const int grp = i / group_items(), t0 = grp * tg, n = min(tg, T - t0);
        return t0 + (i - grp * group_items()) % n;
    }
    __host__ __device__ int unit_of(int i) const {
        if (tile_major) return i % U;
        const int grp = i / group_items(), t0 = grp * tg, n = min(tg, T - t0);
        return (i - grp * group_items()) / n;
    }
    __host__ __device__ int item(int t, int u) const {
        if (tile_major) return t * U + u;
        const int grp = t / tg, t0 = grp * tg, n = min(tg, T - t0);
        return grp * group_items() + u * n + (t - t0);
    }
    __host__ __device__ int first(int c) const { return static_cast<int>(static_cast<long long>(c) * items / G); }
    __host__ __device__ int owner(int i) const {
        return static_cast<int>((static_cast<long long>(i + 1) * G - 1) / items);
    }
    // A share is a run of consecutive items of one CTA within a tile. When the items of tile t
    // are consecutive (tile-major, or a group of one tile) a share starts at unit 0 and at the
    // first item of every CTA that begins inside the tile; otherwise every unit is a share.
    __host__ __device__ bool consecutive(int t) const {
        if (tile_major) return true;
        const int t0 = (t / tg) * tg;
        return min(tg, T - t0) == 1;
    }
    __host__ __device__ int shares(int t) const {
        if (!consecutive(t)) return U;
        const int a0 = item(t, 0);
        return owner(a0 + U - 1) - owner(a0) + 1;
    }
    // units a CTA's share touches (a cyclic range starting at unit_of(first item))
    __host__ __device__ int span(int i0, int i1) const {
        if (i1 <= i0) return 0;
        if (tile_major) return i1 - i0 < U ? i1 - i0 : U;
        const int n_min = T % tg == 0 ? tg : min(tg, T % tg);  // the smallest group
        if (i1 - i0 >= n_min * U) return U;
        // at most one group boundary in between; units rise inside a group and restart at 0
        int d = unit_of(i1 - 1) - unit_of(i0);
        const bool crosses = (i1 - 1) / group_items() != i0 / group_items();
        if (crosses && d >= 0) return U;  // the rest of one group and the start of the next cover every unit
        if (d < 0) d += U;
        return d + 1;
    }
};

// Kernel parameters the loops read, copied once into registers (parameters reached through a
// pointer would be reloaded after every barrier).
struct Ctx {
    Sched sc;
    const void* X;  // activations: fp32 (PN) or bf16 (NVFP4)
    float* Y;
    float* ws;
    uint32_t* cnt;
    int* err;
    int N, K, M, NS, RB;
    unsigned flags;
};

// Next item of a share: (t, u) in the share's order, without divisions.
__device__ __forceinline__ void next_item(const Sched& sc, int& t, int& u) {
    if (sc.tile_major) {
        if (++u == sc.U) {
            u = 0;
            ++t;
        }
        return;
    }
    const int t0 = (t / sc.tg) * sc.tg, t_end = min(t0 + sc.tg, sc.T);
    if (++t == t_end) {
        t = t0;
        if (++u == sc.U) {  // next group
            u = 0;
            t = t_end;
        }
    }
}

// A run: consecutive items of a CTA's share with the same K unit (one item in tile-major order
// unless U = 1). gi = index of its first item within the share.
struct RunCursor {
    int gi, t, u;
};

// Advance to the next run; false when the share has no more items.
__device__ __forceinline__ bool next_run(const Sched& sc, int n_items, RunCursor& rc) {
    const int u_prev = rc.u;
    do {
        next_item(sc, rc.t, rc.u);
        ++rc.gi;
    } while (rc.gi < n_items && rc.u == u_prev);
    return rc.gi < n_items;
}

// One builder warp's loop over the runs of its CTA's share: issue(u, buf) starts the cp.async
// copies of unit u's x rows (this warp's jobs) into x buffer buf, build(slot, buf) turns them
// into the operands of ring slot `slot`. The copies run XB - 1 runs ahead of the build (x loads
// wait behind the weight stream, some microseconds under load). A slot is rebuilt only after
// the consumers released it. False if a wait gave up.
template <int XB, class SM, class Issue, class Build>
__device__ __forceinline__ bool builder_loop(const SM& sm, const Sched& sc, int i0, int n_items, int RB, int lane,
                                             Issue&& issue, Build&& build) {
    RunCursor cur{0, sc.tile_of(i0), sc.unit_of(i0)};
    RunCursor iss = cur;  // the next run to copy
    bool more = true;     // iss is a run of the share
#pragma unroll
    for (int k = 0; k < XB; ++k) {
        if (more) {
            issue(iss.u, k);
            more = next_run(sc, n_items, iss);
        }
        cp_async_commit();  // one group per run (empty past the end)
    }
    for (int r = 0;; ++r) {
        cp_async_wait<XB - 1>();  // group r: the copies of run r have landed
        __syncwarp();
        const int slot = r % RB;
        if (r >= RB && !mbar_wait_warp(sm.op_empty(slot), ((r / RB) - 1) & 1)) return false;
        build(slot, r % XB);
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.op_full(slot));
        if (!next_run(sc, n_items, cur)) return true;
        if (more) {
            issue(iss.u, r % XB);  // run r + XB into the buffer run r used
            more = next_run(sc, n_items, iss);
        }
        cp_async_commit();
    }
}

// Resident mode: the participating warps (index pw of npw) copy the x rows of the CTA's units
// (copy(r) issues row r of n_rows, one warp per row) and then run every build job (job(i),
// i < n_jobs), with a named barrier after each phase. With overlap the x bytes live in weight
// stages that tensor-map copies overwrite next: the generic-proxy reads are fenced first.
template <class CopyF, class JobF>
__device__ __forceinline__ void resident_prologue(int pw, int npw, int n_rows, int n_jobs, bool overlap, CopyF&& copy,
                                                  JobF&& job) {
    griddep_wait();  // X belongs to the previous grid until now
    for (int r = pw; r < n_rows; r += npw) copy(r);
    cp_async_commit();
    cp_async_wait<0>();
    named_sync(1, npw * 32);
    for (int i = pw; i < n_jobs; i += npw) job(i);
    if (overlap) fence_proxy_async_smem();
    named_sync(1, npw * 32);
}

// Consumer side of the ring: at the first item of a new run release the previous run's slot and
// wait for this one's operands. r = the run of the current item (-1 before the first).
template <class SM>
__device__ __forceinline__ bool consumer_next_run(const SM& sm, int RB, int lane, int& r) {
    if (r >= 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.op_empty(r % RB));
    }
    ++r;
    return mbar_wait_warp(sm.op_full(r % RB), (r / RB) & 1);
}

// Y rows t*128 + 4*lane .. + 3 of activation row m.
__device__ __forceinline__ void put_y(const Ctx& a, int t, int m, int lane, float4 v) {
    const int row = t * kTileRows + 4 * lane;
    float* y = a.Y + static_cast<size_t>(m) * a.N;
    if (row + 0 < a.N) y[row + 0] = v.x;
    if (row + 1 < a.N) y[row + 1] = v.y;
    if (row + 2 < a.N) y[row + 2] = v.z;
    if (row + 3 < a.N) y[row + 3] = v.w;
}

// Reducer side of one share of tile t (consecutive items of this CTA, units u_first ..
// u_first+n-1): add the two halves; a whole tile goes to Y, a part to its workspace slot (it is
// counted later). Returns true for a part.
template <int MAXM, class SM>
__device__ __forceinline__ bool reduce_share(const Ctx& a, const SM& sm, int buf, int t, int u_first, int n_units,
                                             int lane) {
    const Sched& sc = a.sc;
    // the two halves' row sums into registers; the buffer goes back to the consumers at once
    const float* part = sm.part();
    float4 v[MAXM];
#pragma unroll
    for (int m = 0; m < MAXM; ++m) {
        if (m < a.M) {
            const float4 p0 = reinterpret_cast<const float4*>(part + ((0 * 2 + buf) * a.M + m) * kPartPitch)[lane];
            const float4 p1 = reinterpret_cast<const float4*>(part + ((1 * 2 + buf) * a.M + m) * kPartPitch)[lane];
            v[m] = make_float4(p0.x + p1.x, p0.y + p1.y, p0.z + p1.z, p0.w + p1.w);
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.part_free(buf));
    if (n_units == sc.U) {
#pragma unroll
        for (int m = 0; m < MAXM; ++m)
            if (m < a.M) put_y(a, t, m, lane, v[m]);
        return false;
    }
    float* slot = a.ws + (static_cast<size_t>(t) * sc.U + u_first) * a.M * kTileRows;
#pragma unroll
    for (int m = 0; m < MAXM; ++m)
        if (m < a.M) __stcg(reinterpret_cast<float4*>(slot + m * kTileRows) + lane, v[m]);
    return true;
}

// Count the np partial shares of this CTA (tiles in pending[]) after their slots were stored:
// the ones that complete their tile are appended to finish[] (n_finish[0] entries). One warp.
template <class SM>
__device__ __forceinline__ void count_shares(const Ctx& a, const SM& sm, int np, int lane) {
    __syncwarp();  // every lane's slot stores come before the (releasing) counts
    int* pend = sm.pending();
    int* fin = sm.finish();
    for (int k0 = 0; k0 < np; k0 += 32) {
        const int k = k0 + lane;
        bool last = false;
        int t = 0;
        if (k < np) {
            t = pend[k];
            last = atomic_add_acq_rel(a.cnt + t, 1u) == static_cast<unsigned>(a.sc.shares(t) - 1);
        }
        const unsigned mask = __ballot_sync(0xffffffffu, last);
        const int base = *sm.n_finish();
        if (last) fin[base + __popc(mask & ((1u << lane) - 1u))] = t;
        __syncwarp();
        if (lane == 0) *sm.n_finish() = base + __popc(mask);
        __syncwarp();
    }
    // the finishers read the other CTAs' slots after the CTA barrier that follows: the acquiring
    // count that completed the tile orders those reads after the other CTAs' releasing counts
}

// Sum the shares of tile t for activation row m in unit order into Y (one warp). The slot
// loads go out eight at a time; the additions keep unit order, so the sum does not depend on
// which CTA finishes the tile. The m == 0 call clears the tile's counter for the next launch
// (no other CTA reads it again in this one).
__device__ __forceinline__ void finish_tile(const Ctx& a, int t, int m, int lane) {
    const Sched& sc = a.sc;
    const bool consec = sc.consecutive(t);
    const int a0 = sc.item(t, 0);
    const int c_lo = consec ? sc.owner(a0) : 0;
    const int n = consec ? sc.owner(a0 + sc.U - 1) - c_lo + 1 : sc.U;  // shares of the tile
    const float* base = a.ws + (static_cast<size_t>(t) * sc.U * a.M + m) * kTileRows;
    auto unit_of_share = [&](int j) { return !consec ? j : (j == 0 ? 0 : sc.first(c_lo + j) - a0); };
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    constexpr int B = 8;  // slot loads in flight per lane
    for (int j0 = 0; j0 < n; j0 += B) {
        float4 v[B];
#pragma unroll
        for (int i = 0; i < B; ++i)
            if (j0 + i < n)
                v[i] = __ldcg(reinterpret_cast<const float4*>(
                                  base + static_cast<size_t>(unit_of_share(j0 + i)) * a.M * kTileRows) + lane);
#pragma unroll
        for (int i = 0; i < B; ++i)
            if (j0 + i < n) {
                acc.x += v[i].x;
                acc.y += v[i].y;
                acc.z += v[i].z;
                acc.w += v[i].w;
            }
    }
    put_y(a, t, m, lane, acc);
    if (m == 0 && lane == 0) a.cnt[t] = 0u;  // ready for the next launch
}

// The tiles this CTA completed, (tile, activation row) pairs spread over all nwarps warps.
template <class SM>
__device__ __forceinline__ void finish_tiles(const Ctx& a, const SM& sm, int warp, int nwarps, int lane) {
    const int nf = *sm.n_finish();
    for (int k = warp; k < nf * a.M; k += nwarps) finish_tile(a, sm.finish()[k / a.M], k % a.M, lane);
}

// ---- host ----------------------------------------------------------------------------------

uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }


}  // namespace
}  // namespace pnq
