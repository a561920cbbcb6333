// pnq_cluster.cuh -- the GEMV pipeline shared by the fast paths (PN on the tensor cores, PN on
// the CUDA cores, NVFP4): work split, weight stream, operand builders, on-chip reduction.
//
// Work split (pnq_split.cuh). Clusters of C = 1 or 2 CTAs own disjoint row ranges; the CTAs of a
// cluster share that range's (K unit, row group) items, unit-major. A stage is up to 64 rows of
// one unit, copied as 8-row pieces by tensor-map copies into a ring of S stages (full / empty
// mbarriers, L2 evict-first).
//
// Warp roles. Eight consumer warps in two groups of four; the stages alternate between the groups
// by the parity of their 64-row block, and warp q of a group takes row group q of the block, so
// every row group belongs to one warp for the whole launch and its partial sums need no lock. One
// producer warp issues the copies; NB builder warps turn x into the operands of each K unit (two
// slots under full / empty mbarriers).
//
// Reduction. Each CTA keeps fp32 partials of its cluster's rows in shared memory; after a cluster
// barrier every CTA sums a slice of the rows over the cluster's CTAs in CTA order (distributed
// shared memory), so the result does not depend on timing, and writes Y. No global workspace.
//
// Launch overlap. griddepcontrol.launch_dependents at entry; with the static-weights flag the
// producer streams weights without waiting for the previous grid; the builders (x) and the Y
// stores wait for it. When a plan fits two CTAs per SM, the next launch's CTA is resident beside
// this one and fills its ring meanwhile.
//
// Bounded waits. Every mbarrier wait gives up after ~2 s of %globaltimer and records a site code
// in the device error word; every role then runs to the common barriers (no trap, no hang).
//
// A format policy F supplies the unit geometry, the copies of one 8-row piece, the operand build
// of one activation row and the multiply of one 16-row group (see PnMma in pnq_gemv_pn.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>

#include "pnq_device.cuh"
#include "pnq_internal.h"
#include "pnq_split.cuh"

namespace pnq {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kStageRows = kStageGroups * kGroupRows;  // 64
constexpr unsigned kStaticWeights = 1u;
constexpr uint32_t kSmemPair = 112u * 1024u;  // two CTAs per SM (228 KB, 1 KB reserved per CTA)
constexpr uint32_t kSmemOne = 226u * 1024u;

// Arguments every fast path shares.
struct ClArgs {
    const void* X;
    float* Y;
    int* err;
    Split sp;
    int N, K, M, S, rc;  // rc: partial rows per activation row (>= any cluster's rows, multiple of 16)
    int xs;              // x slots (units of x prefetched ahead of the operand build), 1..8
    unsigned flags;
    uint32_t off_zb, off_part, off_rec, off_x, off_stage;
};

template <class F>
struct KArgs {
    CUtensorMap map[F::MAPS];  // first: 64-byte aligned in the parameter space
    ClArgs c;
    typename F::Extra e;
};

// Shared-memory regions (offsets from the 1024-aligned base).
template <class F>
struct ClSmem {
    uint8_t* base;
    uint32_t bar0;
    int S, rc;
    uint32_t off_zb, off_part, off_rec, off_x, off_stage;
    __device__ uint32_t full(int s) const { return bar0 + 8u * s; }
    __device__ uint32_t empty(int s) const { return bar0 + 8u * (S + s); }
    __device__ uint32_t bfull(int k) const { return bar0 + 8u * (2 * S + k); }
    __device__ uint32_t bempty(int k) const { return bar0 + 8u * (2 * S + 2 + k); }
    __device__ float* zb(int k) const { return reinterpret_cast<float*>(base + off_zb) + k * F::ZB; }
    __device__ float* part() const { return reinterpret_cast<float*>(base + off_part); }  // [M][rc]
    __device__ uint8_t* rec(int k) const { return base + off_rec + static_cast<uint32_t>(k) * F::REC; }
    __device__ uint8_t* xrow(int slot, int m, int M) const {
        return base + off_x + static_cast<uint32_t>(slot * M + m) * F::UK * F::X_BYTES;
    }
    __device__ uint8_t* stage(int s) const { return base + off_stage + static_cast<uint32_t>(s) * F::STAGE_BYTES; }
};

template <class F>
__global__ void __launch_bounds__(F::THREADS, F::MINB) cluster_gemv_kernel(const __grid_constant__ KArgs<F> ka) {
    constexpr int CW = kConsumerWarps, PRODUCER = CW, BUILDER = CW + 1;
    const ClArgs& a = ka.c;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const ClSmem<F> sm{base, smem_addr(base), a.S, a.rc, a.off_zb, a.off_part, a.off_rec, a.off_x, a.off_stage};
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int M = a.M, S = a.S;
    const Split::Cta ct = a.sp.cta(blockIdx.x);
    const int u_first = ct.i1 > ct.i0 ? static_cast<int>(ct.i0 / ct.Rg) : 0;
    const int n_units = ct.i1 > ct.i0 ? static_cast<int>((ct.i1 - 1) / ct.Rg) - u_first + 1 : 0;

    if (threadIdx.x == 0) {
        griddep_launch_dependents();
        for (int s = 0; s < S; ++s) {
            mbar_init(sm.full(s), 1);
            mbar_init(sm.empty(s), 4);  // the four warps of the consuming group
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(sm.bfull(k), F::NB);
            mbar_init(sm.bempty(k), CW);
        }
        mbar_fence_init();
    }
    // zero the row partials
    {
        float4* p = reinterpret_cast<float4*>(sm.part());
        const int n4 = M * a.rc / 4;
        for (int i = threadIdx.x; i < n4; i += F::THREADS) p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();

    if (warp == PRODUCER) {
        // ---------------- producer: the copies of each 8-row piece of a stage ----------------
        if (lane == 0 && ct.i1 > ct.i0) {
            const uint64_t pol = l2_policy_evict_first();
            if (!(a.flags & kStaticWeights)) griddep_wait();  // W may be written by the previous grid
            bool ok = true;
            StageWalk wk(ct);
            Stage st;
            int s = 0;
            const int pieces_c = ct.rows / kPieceRows;
            for (; ok && wk.next(st); ++s) {
                const int slot = s % S;
                if (s >= S && !mbar_wait_bounded(sm.empty(slot), ((s / S) - 1) & 1)) {
                    ok = false;
                    break;
                }
                const int pc0 = 2 * st.g0, pc1 = min(2 * st.g1, pieces_c);
                mbar_arrive_expect_tx(sm.full(slot), static_cast<uint32_t>((pc1 - pc0) * F::PIECE_TX));
                const uint32_t dst = smem_addr(sm.stage(slot));
                const int row_b = static_cast<int>(ct.row0) + pc0 * kPieceRows;
                if (pc1 - pc0 == 2 * kStageGroups) {
                    // a whole stage: one copy of 64 rows (the copy engine's cost grows with the number
                    // of copies and rows it handles, far more than with bytes)
                    F::issue_stage(ka.map, dst, st.u, row_b, sm.full(slot), pol);
                } else {
                    for (int p = 0; p < pc1 - pc0; ++p)
                        F::issue(ka.map, dst, p, st.u, row_b + p * kPieceRows, sm.full(slot), pol);
                }
            }
            if (!ok) record_error(a.err, kErrEmptyWait);
            // every copy issued has landed before the CTA may exit
            bool drained = true;
            for (int gg = max(0, s - S); drained && gg < s; ++gg)
                drained = mbar_wait_bounded(sm.full(gg % S), (gg / S) & 1);
            if (!drained) record_error(a.err, kErrDrainWait);
        }
        __syncwarp();
    } else if (warp >= BUILDER) {
        // ---------------- builders: operands of each unit; activation rows m = b, b + NB, .. -----------
        if (n_units > 0) {
            griddep_wait();  // X belongs to the previous grid until now
            const int b = warp - BUILDER;
            const uint8_t* X = static_cast<const uint8_t*>(a.X);
            constexpr int ROWB = F::UK * F::X_BYTES;  // bytes of x per row and unit
            const int XS = a.xs;                      // x slots: units whose x is in flight or held
            // x of unit k (this warp's rows) into x slot k % XS, as one cp.async group (possibly
            // empty), so that exactly XS groups are in flight when unit k is waited for
            auto load_x = [&](int k) {
                if (k < n_units) {
                    const int u = u_first + k;
                    for (int m = b; m < M; m += F::NB) {
                        const uint8_t* src = X + (static_cast<size_t>(m) * a.K + static_cast<size_t>(u) * F::UK) * F::X_BYTES;
                        const uint32_t dst = smem_addr(sm.xrow(k % XS, m, M));
                        for (int q = lane; q < ROWB / 16; q += 32) cp_async16(dst + 16u * q, src + 16 * q);
                    }
                }
                cp_async_commit();
            };
            for (int k = 0; k < XS; ++k) load_x(k);
            bool ok = true;
            for (int k = 0; k < n_units && ok; ++k) {
                const int slot = k & 1;
                cp_async_wait_dyn(XS - 1);  // unit k's group has landed
                __syncwarp();
                if (k >= 2 && !mbar_wait_warp(sm.bempty(slot), ((k >> 1) - 1) & 1)) {
                    ok = false;
                    break;
                }
                for (int m = b; m < M; m += F::NB)
                    F::build(sm.rec(slot), sm.zb(slot), sm.xrow(k % XS, m, M), m, ka.e, lane);
                __syncwarp();
                if (lane == 0) mbar_arrive(sm.bfull(slot));
                load_x(k + XS);  // into the slot just read
            }
            cp_async_wait<0>();  // nothing in flight when the warp leaves
            if (!ok && lane == 0) record_error(a.err, kErrOperandWait);
        }
    } else if (warp < CW) {
        // ---------------- consumers ----------------
        const int grp = warp >> 2, q = warp & 3;
        const typename F::Lane ln(lane, M);
        bool ok = true;
        StageWalk wk(ct);
        Stage st;
        int s = 0, k = -1;  // stage index, unit index (from u_first) whose operands are held
        float* part = sm.part();
        for (; ok && wk.next(st); ++s) {
            const int ku = st.u - u_first;
            if (ku != k) {  // a new unit: release the previous operands, wait for the next
                if (k >= 0) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(sm.bempty(k & 1));
                }
                k = ku;
                if (!mbar_wait_warp(sm.bfull(k & 1), (k >> 1) & 1)) {
                    ok = false;
                    k = -1;
                    break;
                }
            }
            if ((st.blk & 1) != grp) continue;
            const int slot = s % S;
            if (!mbar_wait_warp(sm.full(slot), (s / S) & 1)) {
                ok = false;
                break;
            }
            const int gr = st.blk * kStageGroups + q;  // this warp's row group in the cluster
            if (gr >= st.g0 && gr < st.g1) {
                uint8_t* stg = sm.stage(slot);
                const int lg = gr - st.g0;       // the group's position in the stage
                const int lr = gr * kGroupRows;  // first row of the group in the cluster
                if (lr + 8 >= ct.rows) {
                    // the group's second half lies past the cluster's rows and was not copied: zero
                    // it (this warp alone reads it) so that it adds nothing
                    F::zero_half(stg, lg, lane);
                    fence_proxy_async_smem();  // before the stage is refilled by the copy engine
                    __syncwarp();
                }
                typename F::Acc acc;
                F::group(stg, lg, sm.rec(k & 1), sm.zb(k & 1), M, ln, acc);
                F::flush(part, a.rc, lr, sm.zb(k & 1), M, ln, acc);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.empty(slot));
        }
        if (k >= 0) {
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.bempty(k & 1));
        }
        if (!ok && lane == 0) record_error(a.err, kErrFullWait);
    }

    // ---------------- cluster sum of the row partials -> Y ----------------
    __syncthreads();
    const int C = a.sp.C;
    if (C > 1) cluster_sync();
    {
        griddep_wait();  // Y may still be read by the previous grid
        const int rank = blockIdx.x % C;
        const int64_t left_rows = static_cast<int64_t>(a.N) - ct.row0;
        const int rows = left_rows < ct.rows ? static_cast<int>(left_rows) : ct.rows;
        const int E = M * rows;
        const int e0 = static_cast<int>(static_cast<int64_t>(rank) * E / C);
        const int e1 = static_cast<int>(static_cast<int64_t>(rank + 1) * E / C);
        const uint32_t pbase = smem_addr(sm.part());
        for (int e = e0 + threadIdx.x; e < e1; e += F::THREADS) {
            const int m = e / rows, r = e - m * rows;
            float v;
            if (C == 1) {
                v = sm.part()[m * a.rc + r];
            } else {
                const uint32_t off = 4u * static_cast<uint32_t>(m * a.rc + r);
                v = 0.0f;
                for (int j = 0; j < C; ++j) v += ld_dsmem_f32(pbase + off, static_cast<uint32_t>(j));
            }
            a.Y[static_cast<size_t>(m) * a.N + ct.row0 + r] = v;
        }
    }
    if (C > 1) cluster_sync();  // no CTA leaves while another still reads its partials
}

// ---- host side --------------------------------------------------------------------------------------

struct ClPlan {
    Split sp{};
    int S = 0, rc = 0, minb = 1, xs = 1;
    uint32_t off_zb = 0, off_part = 0, off_rec = 0, off_x = 0, off_stage = 0, total = 0;
};

inline uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// Shared-memory layout for S weight stages and XS x slots; the total (without the 1024-byte
// alignment slack).
template <class F>
void cl_layout(int M, int S, int XS, ClPlan& p) {
    p.S = S;
    p.xs = XS;
    p.off_zb = align_up(8u * (2u * S + 4u), 16);
    p.off_part = align_up(p.off_zb + 2u * F::ZB * 4u, 16);
    p.off_rec = align_up(p.off_part + static_cast<uint32_t>(M) * p.rc * 4u, 128);
    p.off_x = align_up(p.off_rec + 2u * F::REC, 16);
    p.off_stage = align_up(p.off_x + static_cast<uint32_t>(XS * M) * F::UK * F::X_BYTES, 1024);
    p.total = p.off_stage + static_cast<uint32_t>(S) * F::STAGE_BYTES;
}

// K units a CTA's share touches.
inline int cl_units(const Split::Cta& t) {
    return t.i1 > t.i0 ? static_cast<int>((t.i1 - 1) / t.Rg - t.i0 / t.Rg) + 1 : 0;
}

// Estimated time of one CTA's share: its bytes at the per-SM share of HBM, the serial work of its
// busiest consumer warp (F::GROUP_S seconds per row group and unit), or the round trips for x
// (XS units in flight, ~0.8 us each), whichever is longest, plus the cluster's final sum.
// per = CTAs of this launch sharing an SM (its HBM share and issue slots); S = weight stages: a
// CTA's stream rate is bounded by the stages in flight (all but the two its consumer groups hold)
// over the loaded HBM latency (~1.8 us).
template <class F>
double cl_cta_cost(const Split& sp, int block, int XS, int per, int S) {
    const Split::Cta t = sp.cta(block);
    StageWalk wk(t);
    Stage st;
    int64_t pieces = 0;
    int per_warp[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    const int pc = t.rows / kPieceRows;
    while (wk.next(st)) {
        pieces += std::min(2 * st.g1, pc) - 2 * st.g0;
        for (int gr = st.g0; gr < st.g1; ++gr) ++per_warp[(st.blk & 1) * 4 + (gr % kStageGroups)];
    }
    int most = 0;
    for (int w : per_warp) most = std::max(most, w);
    const double rate = std::min(42e9 / per, std::max(1, S - 2) * static_cast<double>(F::STAGE_BYTES) / 1.8e-6);
    const double bytes_s = static_cast<double>(pieces) * F::PIECE_TX / rate;
    const double warp_s = most * F::GROUP_S * (per > 1 ? 1.4 : 1.0);
    const double x_s = (cl_units(t) + XS - 1) / XS * 0.8e-6;
    return std::max(std::max(bytes_s, warp_s), x_s) + (sp.C > 1 ? 0.3e-6 : 0.0);
}

// waves > 1: waves * (SMs / C) clusters, for row ranges whose partials would not fit otherwise
inline Split cl_split(int64_t N, int U, int sms, int C, int waves = 1) {
    Split sp;
    sp.pieces = (N + kPieceRows - 1) / kPieceRows;
    sp.U = U;
    sp.C = C;
    sp.ncl = static_cast<int>(std::min<int64_t>(static_cast<int64_t>(sms / C) * waves, sp.pieces));
    return sp;
}

inline int cl_rows_max(const Split& sp) {
    int64_t most = 0;
    for (int c = 0; c < sp.ncl; ++c) most = std::max(most, sp.piece0(c + 1) - sp.piece0(c));
    return static_cast<int>((most * kPieceRows + kGroupRows - 1) / kGroupRows * kGroupRows);
}

// A layout for one CTA per SM (pair = false: up to the whole shared memory) or two (pair = true):
// x slots for as many of the CTA's units as possible (up to 4; then 2, 1), and within that the
// deepest weight ring (kMaxStages..3 stages, or s_req). nu = the most units any CTA of the plan
// touches.
constexpr int kMaxStages = 12;
template <class F>
bool cl_fit_layout(int M, int s_req, int nu, bool pair, ClPlan& q) {
    for (uint32_t budget : {kSmemPair, kSmemOne}) {
        if (budget == kSmemPair && (F::MINB < 2 || !pair)) continue;
        if (budget == kSmemOne && pair) continue;
        for (int xs : {4, 2, 1}) {
            const int XS = std::max(1, std::min(xs, nu));
            for (int S = (s_req > 0 ? s_req : kMaxStages); S >= (s_req > 0 ? s_req : 3); --S) {
                cl_layout<F>(M, S, XS, q);
                if (q.total + 1024u <= budget) {
                    q.minb = (budget == kSmemPair) ? 2 : 1;
                    return true;
                }
            }
        }
    }
    return false;
}

// Cluster size (1 or 2: both spread one CTA per SM over all SMs of the part), CTAs of the launch
// per SM (2 when two fit: twice the warps on the launch's work), clusters and ring depth for one
// shape: the plan with the smallest estimated time. c_req / s_req / k_req > 0 force the cluster
// size, the stages and the CTAs per SM.
template <class F>
bool cl_make_plan(int64_t N, int U, int M, int sms, int c_req, int s_req, int k_req, ClPlan& p) {
    bool found = false;
    double best = 0.0;
    for (int per : {2, 1}) {
        if ((per == 2 && F::MINB < 2) || (k_req > 0 && per != k_req)) continue;
        for (int C : {1, 2}) {
            if (c_req > 0 && C != c_req) continue;
            if (sms / C < 1) continue;
            for (int waves = 1; waves <= 64; ++waves) {
                Split sp = cl_split(N, U, sms * per, C, waves);
                if (static_cast<int64_t>(cl_rows_max(sp) / kGroupRows) * U > INT32_MAX) continue;
                ClPlan q;
                q.sp = sp;
                q.rc = cl_rows_max(sp);
                int nu = 0;
                for (int b = 0; b < sp.ncl * C; ++b) nu = std::max(nu, cl_units(sp.cta(b)));
                if (!cl_fit_layout<F>(M, s_req, nu, per == 2, q)) {
                    if (sp.ncl >= sp.pieces) break;
                    continue;  // more, smaller clusters
                }
                double cost = 0.0;
                for (int b = 0; b < sp.ncl * C; ++b) cost = std::max(cost, cl_cta_cost<F>(sp, b, q.xs, per, q.S));
                cost *= waves;
                if (!found || cost < best * 0.98) {
                    p = q;
                    best = cost;
                    found = true;
                }
                break;
            }
        }
    }
    return found;
}

struct PlanKey {
    const void* kern;
    int M, sms, c, s, k, U;
    int64_t N;
    bool operator<(const PlanKey& o) const {
        return std::tie(kern, M, sms, c, s, k, U, N) < std::tie(o.kern, o.M, o.sms, o.c, o.s, o.k, o.U, o.N);
    }
};

template <class F>
bool cl_cached_plan(int64_t N, int U, int M, int sms, int c_req, int s_req, int k_req, ClPlan& p) {
    static std::mutex mu;
    static std::map<PlanKey, ClPlan> cache;
    const PlanKey key{reinterpret_cast<const void*>(&cl_make_plan<F>), M, sms, c_req, s_req, k_req, U, N};
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) {
            p = it->second;
            return true;
        }
    }
    if (!cl_make_plan<F>(N, U, M, sms, c_req, s_req, k_req, p)) return false;
    std::lock_guard<std::mutex> lock(mu);
    if (cache.size() < 4096) cache.emplace(key, p);
    return true;
}

// Plans and launches one GEMV; ka.map / ka.e / X, Y, err, N, K, M filled by the caller.
template <class F>
cudaError_t cl_launch(KArgs<F>& ka, int64_t N, int U, const int (&req)[3], bool static_weights,
                      cudaStream_t stream) {
    ClPlan p;
    if (!cl_cached_plan<F>(N, U, ka.c.M, device_sm_count(), req[0], req[1], req[2], p)) return cudaErrorNotSupported;
    auto kern = cluster_gemv_kernel<F>;
    static std::atomic<bool> opted[64];  // the attribute is set once per device (threads may race to set it)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!opted[dev].load(std::memory_order_relaxed)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemOne));
        if (e != cudaSuccess) return e;
        opted[dev].store(true, std::memory_order_relaxed);
    }
    ClArgs& a = ka.c;
    a.sp = p.sp;
    a.S = p.S;
    a.rc = p.rc;
    a.xs = p.xs;
    a.flags = static_weights ? kStaticWeights : 0u;
    a.off_zb = p.off_zb;
    a.off_part = p.off_part;
    a.off_rec = p.off_rec;
    a.off_x = p.off_x;
    a.off_stage = p.off_stage;
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(p.sp.ncl * p.sp.C, 1, 1);
    lc.blockDim = dim3(F::THREADS, 1, 1);
    lc.dynamicSmemBytes = p.total + 1024u;
    lc.stream = stream;
    cudaLaunchAttribute attr[2];
    // may begin while the previous grid in the stream finishes (see griddep_wait in the kernel)
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(p.sp.C);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 2;
    return cudaLaunchKernelEx(&lc, kern, ka);
}

// Environment override "cluster,stages,ctas per SM[,path]" (fields 0 = automatic) from variable
// `name`, read once per call site (each fast path keeps its own static copy).
template <int NV>
inline void env_cluster_config(const char* name, int (&v)[NV]) {
    for (int n = 0; n < NV; ++n) v[n] = 0;
    if (const char* e = std::getenv(name)) {
        const char* p = e;
        for (int n = 0; n < NV && *p; ++n) {
            v[n] = static_cast<int>(std::strtol(p, const_cast<char**>(&p), 10));
            if (*p == ',') ++p;
        }
    }
}

}  // namespace
}  // namespace pnq
