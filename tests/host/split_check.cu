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
//     cluster sizes that spread one CTA per SM (1 or 2);
//   - the row-stream plan (rs_plan): its regions are disjoint, aligned and inside one CTA's budget,
//     every row segment's bulk copies are 16-byte aligned and land inside their stage, the
//     segments of a row tile its units in order, and the dealing of (row group, unit) tasks to the
//     consumer warps gives every task to exactly one warp, each warp the same count to within one;
//   - the row streams' cost estimates pick, for the decode-step projections and both NVFP4 shapes,
//     the K-splitting cluster size that timed fastest on a GB300 with every size forced.
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

template <int TYPE, int LR, int NT = 1>
void check_rs_plan(int64_t N, int Ut, int M, int s_req, bool fma = false, int CL = 1, int max_cl = 0) {
    using C = pnq::Cfg<TYPE, NT, LR>;
    char what[160];
    std::snprintf(what, sizeof what, "rows %s N %lld U %d M %d s %d CL %d max %d", TYPE == pnq::kTypePn3t ? "pn3t" : "pn4t",
                  (long long)N, Ut, M, s_req, CL, max_cl);
    pnq::RsPlan p;
    if (!pnq::rs_plan<TYPE, LR, NT>(N, Ut, M, 152, s_req, p, fma, true, CL, max_cl)) return;
    if (fma && NT > 1) FAIL("CUDA-core decode planned for %d tiles", NT);
    ++plans;
    if (p.CL != CL) FAIL("cluster of %d, asked %d", p.CL, CL);
    if (max_cl > 0 && p.G > max_cl) FAIL("%d clusters, %d resident", p.G, max_cl);
    if (1ll * p.G * CL > 152) FAIL("%d CTAs", p.G * CL);
    const int U = (Ut + CL - 1) / CL;  // the most units of a CTA
    if (s_req > 0 && p.S != s_req) FAIL("forced %d stages, planned %d", s_req, p.S);
    if (p.S < 2 || p.S > 8) FAIL("%d stages", p.S);
    if (p.nseg < 1 || p.nseg > U) FAIL("%d segments", p.nseg);
    if (p.total + 1024u > pnq::kSmemOne) FAIL("total %u", p.total);
    if (p.G < 1 || p.G > 152 / CL || p.G > N) FAIL("grid %d", p.G);
    struct R {
        uint64_t lo, hi;
        const char* name;
    };
    if (p.nseg > pnq::kRsMaxSeg) FAIL("%d segments, table of %d", p.nseg, pnq::kRsMaxSeg);
    const bool whole = U <= pnq::kRsWholeUnits;
    if (whole != (p.nseg == 1)) FAIL("%d segments for %d units", p.nseg, U);
    if (whole && p.pitch != pnq::rs_pitch(U * pnq::kUnitBytes)) FAIL("whole-row pitch %d", p.pitch);
    // every CTA of a cluster: its units [r Ut / CL, (r + 1) Ut / CL) tile [0, Ut); its whole rows fit a stage
    for (int r = 0, prev_u = 0; r < CL; ++r) {
        const int ua = r * Ut / CL, ub = (r + 1) * Ut / CL;
        if (ua != prev_u || ub <= ua || ub - ua > U) FAIL("CTA %d of the cluster has units [%d, %d)", r, ua, ub);
        prev_u = ub;
        const int bytes = (ub - ua) * pnq::kUnitBytes, pitch = pnq::rs_pitch(bytes);
        if (whole && 15u * pitch + bytes > p.stage_bytes) FAIL("rows of cluster CTA %d overflow their stage", r);
        if (r == CL - 1 && ub != Ut) FAIL("cluster units end at %d", ub);
    }
    const uint64_t xbytes = (whole && !fma) ? 4ull * pnq::kRsWarps * 2 * C::UK : 4ull * M * U * C::UK;
    const uint64_t nrec = fma ? 0 : U;
    // x either has a region of its own or lies in the ring's slots [x_slot0, S), slot 2 or later
    // (the producer fills those only after every warp has built its operands)
    const bool x_in_ring = p.x_slot0 < p.S;
    if (x_in_ring) {
        if (fma) FAIL("x in the ring with the CUDA-core decode");
        if (p.x_slot0 < 2) FAIL("x in slot %d", p.x_slot0);
        if (p.off_x != p.off_stage + 1ull * p.x_slot0 * p.stage_bytes ||
            p.off_x + xbytes > p.off_stage + 1ull * p.S * p.stage_bytes)
            FAIL("x [%u, +%llu) outside slots %d..%d", p.off_x, (unsigned long long)xbytes, p.x_slot0, p.S);
    } else if (p.x_slot0 != p.S) {
        FAIL("x slot %d of %d stages", p.x_slot0, p.S);
    }
    std::vector<R> r = {{0, 8ull * (2 * p.S + 3), "barriers"},
                        {p.off_rec, p.off_rec + nrec * C::REC, "B operands"},
                        {p.off_zb, p.off_zb + 4ull * nrec * pnq::rs_zb(NT), "zero-point terms"},
                        {p.off_part, p.off_part + 4ull * pnq::kRsWarps * M * p.rows_pad, "row partials"},
                        {p.off_stage, p.off_stage + 1ull * p.S * p.stage_bytes, "stages"}};
    if (!x_in_ring) r.push_back({p.off_x, p.off_x + xbytes, "x rows"});
    if (p.off_rec % 16 || p.off_zb % 16 || p.off_x % 16 || p.off_part % 16 || p.off_stage % 128 ||
        p.stage_bytes % 128)
        FAIL("misaligned region");
    if (p.off_stage + 1ull * p.S * p.stage_bytes != p.total) FAIL("stages end before the total %u", p.total);
    std::sort(r.begin(), r.end(), [](const R& a, const R& b) { return a.lo < b.lo; });
    for (size_t k = 1; k < r.size(); ++k)
        if (r[k].lo < r[k - 1].hi) FAIL("%s overlaps %s", r[k].name, r[k - 1].name);
    // segments tile [0, U) in order; each one's 16 rows fit a stage at an aligned pitch
    int prev = 0;
    for (int j = 0; j < p.nseg; ++j) {
        const int u0 = j * U / p.nseg, u1 = (j + 1) * U / p.nseg;
        if (u0 != prev || u1 <= u0) FAIL("segment %d = [%d, %d)", j, u0, u1);
        prev = u1;
        const int bytes = (u1 - u0) * pnq::kUnitBytes, pitch = pnq::rs_pitch(bytes);
        if (bytes % 16 || pitch % 16 || pitch < bytes || ((pitch / 16) & 1) == 0) FAIL("pitch %d of %d", pitch, bytes);
        if (15u * pitch + bytes > p.stage_bytes) FAIL("segment %d overflows its stage", j);
        if ((u0 * pnq::kUnitBytes) % 16) FAIL("segment %d source misaligned", j);
    }
    if (prev != U) FAIL("segments end at %d", prev);
    // rows of every cluster, and the task dealing of its stages (a CTA with the most units)
    for (int b = 0; b < p.G; ++b) {
        const int64_t r0 = static_cast<int64_t>(b) * N / p.G, r1 = static_cast<int64_t>(b + 1) * N / p.G;
        const int nrows = static_cast<int>(r1 - r0);
        if (nrows < 1 || nrows > p.rows_pad || p.rows_pad % 16) FAIL("CTA %d of %d rows, partials %d", b, nrows, p.rows_pad);
        if (b > 2 && b < p.G - 2 && N > 1000) continue;  // the dealing depends on rows only through the group count
        const int ngroups = (nrows + 15) / 16;
        std::vector<int> owner(static_cast<size_t>(ngroups) * U, -1), count(pnq::kRsWarps, 0);
        std::vector<int> k0(pnq::kRsWarps);
        for (int w = 0; w < pnq::kRsWarps; ++w) k0[w] = w;
        for (int s = 0; s < ngroups * p.nseg; ++s) {
            const int i = s / p.nseg, j = s % p.nseg, u0 = j * U / p.nseg, n = (j + 1) * U / p.nseg - u0;
            for (int w = 0; w < pnq::kRsWarps; ++w) {
                for (int k = k0[w]; k < n; k += pnq::kRsWarps) {
                    int& o = owner[static_cast<size_t>(i) * U + u0 + k];
                    if (o != -1) FAIL("task (%d, %d) dealt twice", i, u0 + k);
                    o = w;
                    ++count[w];
                }
                k0[w] = (k0[w] - n % pnq::kRsWarps + pnq::kRsWarps) % pnq::kRsWarps;
            }
        }
        for (int o : owner)
            if (o < 0) FAIL("a task of CTA %d is dealt to no warp", b);
        const auto mm = std::minmax_element(count.begin(), count.end());
        if (*mm.second - *mm.first > 1) FAIL("CTA %d: warps get %d..%d tasks", b, *mm.first, *mm.second);
    }
}

template <int LR>
void check_nr_plan(int64_t N, int Ut, int M, int CL = 1, int max_cl = 0) {
    char what[128];
    std::snprintf(what, sizeof what, "nvfp4 rows N %lld U %d M %d CL %d max %d", (long long)N, Ut, M, CL, max_cl);
    pnq::NrArgs a{};
    uint32_t total = 0;
    if (!pnq::nr_plan<LR>(N, Ut, M, 152, a, total, CL, max_cl)) return;
    ++plans;
    const int U = (Ut + CL - 1) / CL;  // the most units of a CTA
    if (a.CL != CL) FAIL("cluster of %d, asked %d", a.CL, CL);
    if (max_cl > 0 && a.G > max_cl) FAIL("%d clusters, %d resident", a.G, max_cl);
    if (1ll * a.G * CL > 152) FAIL("%d CTAs", a.G * CL);
    for (int r = 0, prev_u = 0; r < CL; ++r) {
        const int ua = r * Ut / CL, ub = (r + 1) * Ut / CL;
        if (ua != prev_u || ub <= ua || ub - ua > U) FAIL("CTA %d of the cluster has units [%d, %d)", r, ua, ub);
        prev_u = ub;
        if (r == CL - 1 && ub != Ut) FAIL("cluster units end at %d", ub);
    }
    constexpr int REC = 8 * LR * 16;
    if (a.S < 2 || a.S > pnq::kNrMaxStages) FAIL("%d stages", a.S);
    if (total + 1024u > pnq::kNrSmem) FAIL("total %u", total);
    if (a.nseg < 1 || a.nseg > pnq::kNrMaxSeg) FAIL("%d segments", a.nseg);
    struct R {
        uint64_t lo, hi;
        const char* name;
    };
    std::vector<R> r = {{0, 8ull * (2 * a.S + 2), "barriers"},
                        {a.off_rec, a.off_rec + 1ull * U * REC, "B records"},
                        {a.off_so, a.off_so + 4ull * pnq::kNrMaxM * U, "unit scales"},
                        {a.off_x, a.off_x + 2ull * M * U * 256, "x"},
                        {a.off_part, a.off_part + 4ull * pnq::kNrWarps * M * a.rows_pad, "row partials"},
                        {a.off_stage, a.off_stage + 1ull * a.S * a.stage_bytes, "stages"}};
    if (a.off_rec % 16 || a.off_so % 16 || a.off_x % 16 || a.off_part % 16 || a.off_stage % 128 ||
        a.stage_bytes % 128 || a.scale_region % 16)
        FAIL("misaligned region");
    if (r.back().hi != total) FAIL("stages end at %llu, total %u", (unsigned long long)r.back().hi, total);
    std::sort(r.begin(), r.end(), [](const R& x, const R& y) { return x.lo < y.lo; });
    for (size_t k = 1; k < r.size(); ++k)
        if (r[k].lo < r[k - 1].hi) FAIL("%s overlaps %s", r[k].name, r[k - 1].name);
    int prev = 0;
    for (int j = 0; j < a.nseg; ++j) {
        const int u0 = j * U / a.nseg, u1 = (j + 1) * U / a.nseg, n = u1 - u0;
        if (u0 != prev || n < 1) FAIL("segment %d", j);
        prev = u1;
        const int pc = pnq::nr_pitch(128 * n), ps = pnq::nr_pitch(16 * n);
        if ((pc / 16) % 2 == 0 || (ps / 16) % 2 == 0) FAIL("pitch %d / %d", pc, ps);
        if (15u * pc + 128u * n > a.scale_region) FAIL("codes of segment %d overflow", j);
        if (a.scale_region + 15u * ps + 16u * n > a.stage_bytes) FAIL("scales of segment %d overflow", j);
    }
    if (prev != U) FAIL("segments end at %d", prev);
    for (int b = 0; b < a.G; ++b) {
        const int64_t r0 = static_cast<int64_t>(b) * N / a.G, r1 = static_cast<int64_t>(b + 1) * N / a.G;
        if (r1 - r0 < 1 || r1 - r0 > a.rows_pad) FAIL("CTA %d rows", b);
    }
}

template <int TYPE>
void run_rows() {
    for (int64_t N : {1, 7, 16, 17, 151, 152, 153, 777, 1024, 5120, 12288, 17408, 151936})
        for (int U : {1, 2, 7, 8, 9, 12, 16, 17, 25, 33, 34, 48, 68})
            for (int s : {0, 2, 3, 5})
                for (int M = 1; M <= 8 && !failures; ++M) {
                    for (bool fma : {false, true}) {
                        for (int CL : {1, 2, 4, 8})
                            for (int mc : {0, 17, 36}) {
                                if (CL == 1 && mc) continue;
                                if (M == 1) check_rs_plan<TYPE, 8>(N, U, M, s, fma, CL, mc);
                                if (M == 2) check_rs_plan<TYPE, 16>(N, U, M, s, fma, CL, mc);
                                if (M == 3) check_rs_plan<TYPE, 24>(N, U, M, s, fma, CL, mc);
                                if (M == 4) check_rs_plan<TYPE, 32>(N, U, M, s, fma, CL, mc);
                                if (M > 4) check_rs_plan<TYPE, 32, 2>(N, U, M, s, fma, CL, mc);
                            }
                    }
                }
    // the decode-step projections at M = 1 take the row-stream path
    for (int64_t N : {1024, 5120, 12288, 17408})
        for (int U : {8, 10, 12, 34}) {
            pnq::RsPlan p;
            if (!pnq::rs_plan<TYPE, 8>(N, U, 1, 152, 0, p)) {
                const char* what = "rows plan";
                FAIL("N %lld U %d M 1 has no row-stream plan", (long long)N, U);
            }
        }
}

}  // namespace

// The planner's choice of K-splitting cluster size for the decode-step projections and both NVFP4
// shapes, with the resident-cluster counts of a GB300 at ~210 KB per CTA (76 / 36 / 15 clusters
// of 2 / 4 / 8): the sizes that timed fastest with every size forced.
void check_cluster_choices() {
    auto resident = [](int CL, const pnq::RsPlan&) { return CL == 2 ? 76 : CL == 4 ? 36 : 15; };
    struct Pn {
        int type, M, U;
        int64_t N;
        int want;
    };
    const Pn pn[] = {{pnq::kTypePn3t, 1, 8, 12288, 1},  {pnq::kTypePn4t, 1, 10, 1024, 1},
                     {pnq::kTypePn4t, 1, 12, 5120, 1},  {pnq::kTypePn3t, 1, 8, 17408, 1},
                     {pnq::kTypePn4t, 1, 34, 5120, 4},  {pnq::kTypePn4t, 2, 34, 5120, 4},
                     {pnq::kTypePn3t, 4, 8, 17408, 1},  {pnq::kTypePn4t, 4, 12, 5120, 2},
                     {pnq::kTypePn4t, 4, 10, 1024, 2},  {pnq::kTypePn4t, 4, 34, 5120, 4}};
    for (const Pn& c : pn) {
        char what[96];
        std::snprintf(what, sizeof what, "cluster choice type %d M %d N %lld U %d", c.type, c.M, (long long)c.N, c.U);
        pnq::RsPlan p;
        bool ok = false;
        if (c.type == pnq::kTypePn3t) {
            ok = c.M == 1   ? pnq::rs_best_plan<pnq::kTypePn3t, 8, 1>(c.N, c.U, c.M, 152, 0, false, true, 0, p, resident)
                 : c.M == 2 ? pnq::rs_best_plan<pnq::kTypePn3t, 16, 1>(c.N, c.U, c.M, 152, 0, false, true, 0, p, resident)
                            : pnq::rs_best_plan<pnq::kTypePn3t, 32, 1>(c.N, c.U, c.M, 152, 0, false, true, 0, p, resident);
        } else {
            ok = c.M == 1   ? pnq::rs_best_plan<pnq::kTypePn4t, 8, 1>(c.N, c.U, c.M, 152, 0, false, true, 0, p, resident)
                 : c.M == 2 ? pnq::rs_best_plan<pnq::kTypePn4t, 16, 1>(c.N, c.U, c.M, 152, 0, false, true, 0, p, resident)
                            : pnq::rs_best_plan<pnq::kTypePn4t, 32, 1>(c.N, c.U, c.M, 152, 0, false, true, 0, p, resident);
        }
        ++plans;
        if (!ok) FAIL("no plan");
        else if (p.CL != c.want) FAIL("clusters of %d, the fastest measured were %d", p.CL, c.want);
    }
    struct Nv {
        int M;
        int64_t N;
        int K, want;
    };
    const Nv nv[] = {{1, 17408, 5120, 1}, {1, 5120, 17408, 4}, {2, 17408, 5120, 1}, {2, 5120, 17408, 4},
                     {4, 17408, 5120, 2}, {4, 5120, 17408, 4}, {8, 17408, 5120, 2}, {8, 5120, 17408, 8}};
    for (const Nv& c : nv) {
        char what[96];
        std::snprintf(what, sizeof what, "nvfp4 cluster choice M %d N %lld K %d", c.M, (long long)c.N, c.K);
        const int U = c.K / 256;
        double best = 0.0;
        int pick = 0;
        for (int CL : {1, 2, 4, 8}) {
            pnq::NrArgs a{};
            uint32_t t = 0;
            const int mc = CL == 2 ? 76 : CL == 4 ? 36 : CL == 8 ? 15 : 0;
            const bool ok = c.M == 1   ? pnq::nr_plan<4>(c.N, U, c.M, 152, a, t, CL, mc)
                            : c.M == 2 ? pnq::nr_plan<8>(c.N, U, c.M, 152, a, t, CL, mc)
                            : c.M == 4 ? pnq::nr_plan<16>(c.N, U, c.M, 152, a, t, CL, mc)
                                       : pnq::nr_plan<32>(c.N, U, c.M, 152, a, t, CL, mc);
            if (!ok) continue;
            const double cost = pnq::nr_cost(a, c.N, U, c.M);
            if (pick == 0 || cost < best) {
                best = cost;
                pick = CL;
            }
        }
        ++plans;
        if (pick != c.want) FAIL("clusters of %d, the fastest measured were %d", pick, c.want);
    }
}

int main() {
    check_cluster_choices();
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
    run_rows<pnq::kTypePn3t>();
    run_rows<pnq::kTypePn4t>();
    for (int64_t N : {1, 9, 151, 152, 1000, 5120, 17408, 151936})
        for (int U : {1, 2, 4, 20, 21, 40, 68, 100})
            for (int CL : {1, 2, 4, 8})
                for (int mc : {0, 15, 36}) {
                    if (CL == 1 && mc) continue;
                    check_nr_plan<4>(N, U, 1, CL, mc);
                    check_nr_plan<8>(N, U, 2, CL, mc);
                    check_nr_plan<12>(N, U, 3, CL, mc);
                    check_nr_plan<16>(N, U, 4, CL, mc);
                    for (int M = 5; M <= 8; ++M) check_nr_plan<32>(N, U, M, CL, mc);
                }
    if (failures) return 1;
    std::printf("ok %ld plans, %ld splits\n", plans, splits);
    return 0;
}
