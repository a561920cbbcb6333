// Host check of the fast paths' work split and launch planner (pnq_split.cuh, cl_make_plan in
// pnq_cluster.cuh, with the PN and NVFP4 format policies), against brute force, for many shapes,
// batch widths and forced cluster sizes and stage counts:
//   - the clusters' row ranges tile [0, pieces) in order, each with at least one piece;
//   - inside a cluster the CTAs' items tile [0, row groups x units) in order;
//   - the stage walk of a CTA visits exactly its items, in order, each stage inside one unit and
//     one block of four row groups, and the pieces it copies lie inside the cluster's rows;
//   - a row group always falls to the same consumer warp (block parity, position in the block);
//   - every plan keeps its shared-memory regions (barriers, per-unit terms, row partials, B
//     operand slots, x slots, weight stages) disjoint, aligned and inside the per-CTA budget it
//     claims (two CTAs per SM or one), sizes the partials for the widest cluster, and uses only
//     cluster sizes that spread one CTA per SM (1 or 2).
// Host code only: the kernels are compiled but never launched.
#include "pnq_gemv_pn.cu"
#include "pnq_gemv_nvfp4.cu"

#include <algorithm>
#include <cstdio>
#include <vector>

namespace pnq {
// the planner's translation unit refers to these; the check never calls them
int device_sm_count() { return 152; }
bool encode_u32_map(CUtensorMap*, const void*, int64_t, int64_t, int, int, bool) { return false; }
}  // namespace pnq

namespace {

int failures = 0;
long splits = 0, plans = 0;

#define FAIL(...)                                  \
    do {                                           \
        if (failures++ < 5) {                      \
            std::printf("FAIL %s: ", what);        \
            std::printf(__VA_ARGS__);              \
            std::printf("\n");                     \
        }                                          \
        return;                                    \
    } while (0)

void check_split(const pnq::Split& sp, const char* what) {
    ++splits;
    if (sp.ncl < 1 || sp.ncl > sp.pieces) FAIL("%d clusters for %lld pieces", sp.ncl, (long long)sp.pieces);
    int64_t expect_p = 0;
    for (int c = 0; c < sp.ncl; ++c) {
        const int64_t p0 = sp.piece0(c), p1 = sp.piece0(c + 1);
        if (p0 != expect_p || p1 <= p0) FAIL("cluster %d pieces [%lld, %lld)", c, (long long)p0, (long long)p1);
        expect_p = p1;
        int64_t expect_i = 0;
        std::vector<int> owner;  // consumer warp of each row group
        for (int r = 0; r < sp.C; ++r) {
            const pnq::Split::Cta t = sp.cta(c * sp.C + r);
            if (t.row0 != p0 * pnq::kPieceRows || t.rows != (p1 - p0) * pnq::kPieceRows)
                FAIL("cluster %d rank %d rows %lld+%d", c, r, (long long)t.row0, t.rows);
            if (t.Rg != (t.rows + 15) / 16) FAIL("row groups %d for %d rows", t.Rg, t.rows);
            if (owner.empty()) owner.assign(t.Rg, -1);
            if (t.i0 != expect_i || t.i1 < t.i0) FAIL("cluster %d rank %d items [%lld, %lld)", c, r, (long long)t.i0,
                                                      (long long)t.i1);
            expect_i = t.i1;
            pnq::StageWalk wk(t);
            pnq::Stage st;
            int64_t i = t.i0;
            const int pc = t.rows / pnq::kPieceRows;
            while (wk.next(st)) {
                if (st.g1 <= st.g0 || st.u < 0 || st.u >= sp.U) FAIL("stage u %d groups [%d, %d)", st.u, st.g0, st.g1);
                if (static_cast<int64_t>(st.u) * t.Rg + st.g0 != i) FAIL("stage starts at item %lld, expected %lld",
                                                                          (long long)(st.u * (int64_t)t.Rg + st.g0),
                                                                          (long long)i);
                if (st.blk != st.g0 / pnq::kStageGroups || (st.g1 - 1) / pnq::kStageGroups != st.blk || st.g1 > t.Rg)
                    FAIL("stage groups [%d, %d) block %d of %d groups", st.g0, st.g1, st.blk, t.Rg);
                const int pc1 = std::min(2 * st.g1, pc);
                if (pc1 <= 2 * st.g0 || pc1 - 2 * st.g0 > pnq::kStageGroups * 2)
                    FAIL("stage copies pieces [%d, %d) of %d", 2 * st.g0, pc1, pc);
                for (int gr = st.g0; gr < st.g1; ++gr) {
                    const int w = (st.blk & 1) * 4 + gr % pnq::kStageGroups;
                    if (owner[gr] >= 0 && owner[gr] != w) FAIL("row group %d on warps %d and %d", gr, owner[gr], w);
                    owner[gr] = w;
                }
                i += st.g1 - st.g0;
            }
            if (i != t.i1) FAIL("walk ended at item %lld, share ends at %lld", (long long)i, (long long)t.i1);
        }
        if (expect_i != static_cast<int64_t>((p1 - p0) * pnq::kPieceRows + 15) / 16 * sp.U)
            FAIL("cluster %d items end at %lld", c, (long long)expect_i);
    }
    if (expect_p != sp.pieces) FAIL("pieces end at %lld of %lld", (long long)expect_p, (long long)sp.pieces);
}

template <class Pol>
void check_plan(const char* name, int64_t N, int U, int M, int c_req, int s_req) {
    using Cf = Pol;
    char what[160];
    std::snprintf(what, sizeof what, "%s M %d N %lld U %d C %d S %d", name, M, (long long)N, U, c_req, s_req);
    pnq::ClPlan p;
    if (!pnq::cl_make_plan<Pol>(N, U, M, 152, c_req, s_req, 0, p)) {
        if (c_req == 0 && s_req == 0) FAIL("no plan");
        return;
    }
    ++plans;
    check_split(p.sp, what);
    if (failures) return;
    if (p.sp.C != 1 && p.sp.C != 2) FAIL("cluster of %d", p.sp.C);
    if (c_req > 0 && p.sp.C != c_req) FAIL("forced cluster %d, planned %d", c_req, p.sp.C);
    if (s_req > 0 && p.S != s_req) FAIL("forced %d stages, planned %d", s_req, p.S);
    if (p.S < 3 || p.S > pnq::kMaxStages) FAIL("%d stages", p.S);
    if (p.xs < 1 || p.xs > 8) FAIL("%d x slots", p.xs);
    // one or two CTAs per SM (two only in the pair budget), in whole waves when a wide cluster's
    // partials would not fit otherwise
    const int slots = 152 * p.minb;
    if (p.sp.ncl * p.sp.C > slots && (p.sp.ncl % (slots / p.sp.C) != 0 && p.sp.ncl != p.sp.pieces))
        FAIL("grid %d", p.sp.ncl * p.sp.C);
    for (int c = 0; c < p.sp.ncl; ++c) {
        const int rows = static_cast<int>((p.sp.piece0(c + 1) - p.sp.piece0(c)) * pnq::kPieceRows);
        if ((rows + 15) / 16 * 16 > p.rc) FAIL("cluster %d of %d rows, partials for %d", c, rows, p.rc);
    }
    if (p.rc % 16) FAIL("partial rows %d", p.rc);
    const uint32_t budget = p.minb == 2 ? pnq::kSmemPair : pnq::kSmemOne;
    if (p.minb == 2 && Cf::MINB != 2) FAIL("two CTAs per SM planned for a kernel bounded to one");
    if (p.total + 1024u > budget) FAIL("total %u + 1024 over %u", p.total, budget);
    struct R {
        uint64_t lo, hi;
        const char* name;
    };
    std::vector<R> r = {{0, 8ull * (2 * p.S + 4), "barriers"},
                        {p.off_zb, p.off_zb + 2ull * Cf::ZB * 4, "zero-point terms"},
                        {p.off_part, p.off_part + 4ull * M * p.rc, "row partials"},
                        {p.off_rec, p.off_rec + 2ull * Cf::REC, "B operands"},
                        {p.off_x, p.off_x + 1ull * Cf::X_BYTES * p.xs * M * Cf::UK, "x rows"},
                        {p.off_stage, p.off_stage + static_cast<uint64_t>(p.S) * Cf::STAGE_BYTES, "stages"}};
    if (p.off_zb % 16 || p.off_part % 16 || p.off_rec % 128 || p.off_x % 16 || p.off_stage % 1024)
        FAIL("misaligned region");
    if (r.back().hi != p.total) FAIL("stages end at %llu, total %u", (unsigned long long)r.back().hi, p.total);
    std::sort(r.begin(), r.end(), [](const R& a, const R& b) { return a.lo < b.lo; });
    for (size_t k = 1; k < r.size(); ++k)
        if (r[k].lo < r[k - 1].hi) FAIL("%s overlaps %s", r[k].name, r[k - 1].name);
}

template <int TYPE>
void run_type() {
    const int64_t Ns[] = {1, 7, 8, 9, 16, 17, 100, 128, 1000, 1024, 1217, 5120, 12288, 17408, 50000, 151936};
    const int Us[] = {1, 2, 3, 8, 10, 12, 34, 68};
    for (int64_t N : Ns)
        for (int U : Us)
            for (int M = 1; M <= 16 && !failures; ++M)
                for (int c : {0, 1, 2})
                    for (int s : {0, 3, 6, 12}) {
                        const int nt = (2 * M + 7) / 8;
                        const char* nm = TYPE == pnq::kTypePn3t ? "pn3t" : "pn4t";
                        if (nt == 1) check_plan<pnq::PnMma<TYPE, 1>>(nm, N, U, M, c, s);
                        else if (nt == 2) check_plan<pnq::PnMma<TYPE, 2>>(nm, N, U, M, c, s);
                        else check_plan<pnq::PnMma<TYPE, 4>>(nm, N, U, M, c, s);
                        if (TYPE == pnq::kTypePn3t) {  // NVFP4 over the same (N, units) grid
                            if (M <= 8) check_plan<pnq::NvMma<1>>("nvfp4", N, U, M, c, s);
                            else check_plan<pnq::NvMma<2>>("nvfp4", N, U, M, c, s);
                        }
                    }
}

}  // namespace

int main() {
    // the split alone, over grids the planner does not pick
    for (int64_t N : {1, 8, 9, 63, 64, 65, 1000, 5120, 17408})
        for (int U : {1, 3, 34})
            for (int sms : {1, 2, 3, 7, 76, 152, 300})
                for (int C : {1, 2}) {
                    char what[96];
                    std::snprintf(what, sizeof what, "split N %lld U %d sms %d C %d", (long long)N, U, sms, C);
                    if (sms / C < 1) continue;
                    check_split(pnq::cl_split(N, U, sms, C), what);
                }
    run_type<pnq::kTypePn3t>();
    run_type<pnq::kTypePn4t>();
    if (failures) return 1;
    std::printf("ok %ld plans, %ld splits\n", plans, splits);
    return 0;
}
