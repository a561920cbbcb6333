// Host check of the PN fast path's launch planner (make_plan in pnq_gemv_pn.cu): for many
// shapes, batch widths and forced configurations, every plan the planner accepts must keep its
// shared-memory regions (barriers, share lists, row sums, x, operand slots, weight stages)
// disjoint, aligned and inside the 227 KB limit, give every CTA's share a list entry, size the
// resident operand slots for the widest share, and flag the workspace exactly when a row tile is
// shared by two CTAs. Host code only: the kernels are compiled but never launched.
#include "pnq_gemv_pn.cu"

#include "plan_check.h"

namespace pnq {
// the planner's translation unit refers to these; the check never calls them
int device_sm_count() { return 152; }
bool encode_u32_map(CUtensorMap*, const void*, int64_t, int64_t, int, int, bool) { return false; }
cudaError_t stream_workspace(cudaStream_t, size_t, size_t, float**, uint32_t**) { return cudaErrorNotSupported; }
}  // namespace pnq

namespace {

long rejected = 0;

template <int TYPE, int NT, int TPW>
void run(int M) {
    using C = pnq::Cfg<TYPE, NT, TPW>;
    constexpr int blk = pnq::PnFmt<TYPE>::BLK;
    const int64_t Ns[] = {1, 100, 128, 1000, 1024, 5120, 12288, 17408, 50000, 151936};
    const int64_t Us[] = {1, 2, 3, 8, 10, 12, 34, 68};
    const int grids[] = {0, 1, 3, 7, 13, 40, 152};
    const int nss[] = {0, 2, 3, 4, 6, 8};
    const int rbs[] = {0, 2, 3};
    const int orders[] = {0, 1, 2};
    char what[160];
    for (int64_t N : Ns)
        for (int64_t U : Us)
            for (int grid : grids)
                for (int ns : nss)
                    for (int rb : rbs)
                        for (int order : orders) {
                            const int64_t T = (N + pnq::kTileRows - 1) / pnq::kTileRows;
                            const int cap = grid > 0 ? std::min(grid, 152) : 152;
                            pnq::Plan p;
                            if (!pnq::make_plan(C::UK, C::bfu(M), M, C::NB, T, U, cap, grid > 0, ns, rb, order, p)) {
                                ++rejected;
                                continue;
                            }
                            std::snprintf(what, sizeof what,
                                          "type %d NT %d TPW %d M %d N %lld K %lld grid %d ns %d rb %d order %d", TYPE,
                                          NT, TPW, M, (long long)N, (long long)(U * 8 * blk), grid, ns, rb, order);
                            const uint64_t jobs = static_cast<uint64_t>(M) * (M < C::NB ? 2 : 1);
                            plan_check::Shape s{M,
                                                8ull * C::bfu(M) + 9ull * M * 4,
                                                C::UK * 4ull,
                                                jobs * C::UK * 4ull,
                                                static_cast<uint64_t>(pnq::kStageBytes),
                                                true};
                            plan_check::check_plan(p, s, pnq::kSmemLimit, pnq::kResident, pnq::kXOverlap,
                                                   pnq::kPartPitch, what);
                            if (plan_check::failures) return;
                        }
}

template <int TYPE>
void run_type() {
    for (int M = 1; M <= 16 && !plan_check::failures; ++M) {
        const int nt = (2 * M + 7) / 8;  // the launcher's n8 tiles for M rows
        if (nt == 1) {
            run<TYPE, 1, 1>(M);
            run<TYPE, 1, 2>(M);
        } else if (nt == 2) {
            run<TYPE, 2, 1>(M);
            run<TYPE, 2, 2>(M);
        } else {
            run<TYPE, 4, 1>(M);
            run<TYPE, 4, 2>(M);
        }
    }
}

}  // namespace

int main() {
    run_type<pnq::kTypePn3t>();
    run_type<pnq::kTypePn4t>();
    if (plan_check::failures) return 1;
    std::printf("ok %ld plans (%ld configurations rejected)\n", plan_check::plans, rejected);
    return 0;
}
