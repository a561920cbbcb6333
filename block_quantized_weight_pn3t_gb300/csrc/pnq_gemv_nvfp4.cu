// pnq_gemv_nvfp4.cu -- NVFP4 (W4A16) GEMV on the tensor cores with mma.sync, sm_103a (fast path).
//
// Computes Y[m][n] = sum_k w[n][k] x[m][k] for 1 <= M <= 16 with w = e2m1(code) * e4m3(scale) * g
// ("Quantisation and profiles", NVFP4; tensor-formats page, NVFP4 / E2M1 / E4M3FN): codes two per
// byte, low nibble = even k, one E4M3FN scale per 16 weights along K, one fp32 global multiplier;
// x is bf16. The weights are decoded in registers just before the multiply.
//
// Work split: the stream-K items of pnq_streamk.cuh, here 128 rows x one K unit of 256 weights
// (128 code bytes and 16 scale bytes per row), tile-major.
//
// Memory pipeline. A producer thread loads one item per stage with two tensor-map copies: the
// codes (128 rows x 128 bytes, with the 128-byte swizzle: 16-byte chunk c of row r lands at chunk
// c ^ (r % 8), so the eight rows a warp reads at once fall in different banks) and the scales
// (128 rows x 16 bytes). NS stages under full / empty mbarriers, L2 evict-first.
//
// Decode and multiply. Warp = TPW tiles of 16 rows x half a unit (16 code words per row). Lane
// (g, c) owns code words c, c + 4, c + 8, c + 12 of the half for rows g and g + 8: each word holds
// 8 codes of one scale group. A byte (two codes) becomes an f16x2 A register with
// cvt.rn.f16x2.e2m1x2 and one HMUL2 by the group's scale (cvt.rn.f16x2.e4m3x2): the product of an
// e2m1 and an e4m3 value is exact in fp16. Byte b of words c + 8q and c + 8q + 4 are slice 4q + b
// of the half; B column m holds the matching x pairs of activation row m, scaled by 2^sigma (per
// CTA and row, so that max|x| * 2^sigma lies in [2^14, 2^15)). A bf16 value scaled so is exact in
// fp16 down to 2^-14 (8 significant bits < 11); below that it rounds at 2^-24, 2^-38 of the row's
// largest |x|. The B fragments of a K unit are made by builder warps (sigma per unit and row);
// two accumulator chains (even and odd slices) per tile; each item's sums are scaled by
// g * 2^-sigma of its unit.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>

#include "pnq_device.cuh"
#include "pnq_internal.h"
#include "pnq_streamk.cuh"

namespace pnq {
namespace {

constexpr int kUnitK = 256;                               // weights of a row per K unit
constexpr int kCodeRow = kUnitK / 2;                      // code bytes of a row per unit (128)
constexpr int kScaleRow = kUnitK / 16;                    // scale bytes of a row per unit (16)
constexpr int kCodeBox = kTileRows * kCodeRow;            // 16384
constexpr int kStageBytes = kCodeBox + kTileRows * kScaleRow;  // 18432, a multiple of 1024
constexpr int kSlices = 8;                                // k16 slices per half-unit

template <int NT, int TPW>
struct NvCfg {
    static constexpr int TG = 8 / TPW;            // tile groups per half
    static constexpr int CW = 2 * TG;             // consumer warps
    static constexpr int NB = (TPW == 1) ? 2 : 6;  // builder warps (within the register budget)
    static constexpr int PRODUCER = CW, REDUCER = CW + 1, BUILDER = CW + 2;
    static constexpr int THREADS = 32 * (CW + 2 + NB);
    static constexpr int BFU = NT * 16 * 256;     // fragment bytes per unit: 16 slices x 32 lanes x 8 B per n8 tile
};

struct NvArgs {
    CUtensorMap codes_map;   // codes as u32 [N][K/8], box {32, 128}, 128-byte swizzle
    CUtensorMap scales_map;  // scales as u32 [N][K/64], box {4, 128}
    const uint16_t* X;
    float* Y;
    float* ws;
    uint32_t* cnt;
    int* err;
    Sched sc;
    int N, K, M, NS, RB, XB;
    int x_stage;     // resident mode with x in the weight stages: the first stage holding x
    int pf;          // static weights: stages requested before griddepcontrol.wait
    unsigned flags;  // kStaticWeights, kResident, kXOverlap
    float g;
    uint32_t list_off, part_off, xs_off, ring_off, stage_off, slot_bytes;
    int list_cap;
};

// Shared-memory regions (offsets from the 1024-aligned base): barriers at 0, lists, row sums,
// x buffers, operand slots (a ring, or one per unit of the share in resident mode), weight
// stages. x buffer b (or unit slot b in resident mode) = [M][256] bf16, possibly inside the last
// weight stages.
struct NvSmem {
    uint8_t* base;
    uint32_t bar0;
    int NS, RB, M;
    uint32_t list_off, part_off, xs_off, ring_off, stage_off, slot_bytes;
    int list_cap;
    __device__ uint32_t full(int s) const { return bar0 + 8u * s; }
    __device__ uint32_t empty(int s) const { return bar0 + 8u * (NS + s); }
    __device__ uint32_t op_full(int s) const { return bar0 + 8u * (2 * NS + s); }
    __device__ uint32_t op_empty(int s) const { return bar0 + 8u * (2 * NS + RB + s); }
    __device__ uint32_t part_full(int b) const { return bar0 + 8u * (2 * NS + 2 * RB + b); }
    __device__ uint32_t part_free(int b) const { return bar0 + 8u * (2 * NS + 2 * RB + 2 + b); }
    __device__ uint32_t x_free() const { return bar0 + 8u * (2 * NS + 2 * RB + 4); }
    __device__ float* part() const { return reinterpret_cast<float*>(base + part_off); }
    __device__ uint16_t* xs(int buf) const {  // [M][256] bf16 x rows of one K unit
        return reinterpret_cast<uint16_t*>(base + xs_off) + static_cast<size_t>(buf) * M * kUnitK;
    }
    __device__ uint8_t* slot(int s) const { return base + ring_off + static_cast<uint32_t>(s) * slot_bytes; }
    template <int NT>
    __device__ float* slot_so(int s) const {  // [M] g * 2^-sigma
        return reinterpret_cast<float*>(slot(s) + NvCfg<NT, 1>::BFU);
    }
    __device__ uint8_t* stage(int s) const { return base + stage_off + static_cast<uint32_t>(s) * kStageBytes; }
    __device__ int* n_finish() const { return reinterpret_cast<int*>(base + list_off); }
    __device__ int* pending() const { return reinterpret_cast<int*>(base + list_off) + 4; }
    __device__ int* finish() const { return reinterpret_cast<int*>(base + list_off) + 4 + list_cap; }
};

// Operands of activation row m for one K unit (one builder warp): sigma from the row's largest
// |x| over the unit, the B fragments (column m) and g * 2^-sigma. xr = the row's 256 bf16 x
// values in shared memory. Lane (P, c) = (lane / 4, lane % 4) builds the record of slices
// S = 2P, 2P + 1 (half S / 8, q = (S % 8) / 4, byte b = S % 4): register r holds the x pair at
// k = 8 * (16 * half + c + 8q + 4r) + 2b; 16-byte record [b0, b1 of 2P; b0, b1 of 2P + 1] in the
// lane of B column m.
template <int NT>
__device__ __forceinline__ void nv_build_row(uint8_t* slot_b, float* slot_so, const uint16_t* xr, int m, float g,
                                             int lane) {
    const uint4 xv = reinterpret_cast<const uint4*>(xr)[lane];
    const uint32_t w[4] = {xv.x, xv.y, xv.z, xv.w};
    uint32_t mx = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) mx = max(mx, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
    const uint32_t bits = __reduce_max_sync(0xffffffffu, mx) << 16;  // the fp32 bits of max |x|
    const int E = static_cast<int>(bits >> 23);
    int sg = (bits == 0 || E >= 255) ? 0 : 141 - E;  // max < 2^(E-126)
    sg = min(100, max(-100, sg));
    const float si = exp2i(sg);
    const int P = lane >> 2, c = lane & 3;
    const uint32_t* x32 = reinterpret_cast<const uint32_t*>(xr);
    uint32_t v[4];
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {  // q4 = 2 * (slice - 2P) + register
        const int S = 2 * P + (q4 >> 1), r = q4 & 1;
        const int half = S >> 3, q = (S >> 2) & 1, b = S & 3;
        const uint32_t pair = x32[4 * (16 * half + c + 8 * q + 4 * r) + b];
        const float v0 = __uint_as_float(pair << 16) * si;          // low bf16
        const float v1 = __uint_as_float(pair & 0xFFFF0000u) * si;  // high bf16
        v[q4] = f32x2_to_f16x2(v0, v1);
    }
    uint8_t* tb = slot_b + (m >> 3) * 4096 + P * 512;
    *reinterpret_cast<uint4*>(tb + ((((m & 7) << 2) | c) * 16)) = make_uint4(v[0], v[1], v[2], v[3]);
    if (lane == 0) slot_so[m] = exp2i(-sg) * g;
}

// One half-unit H of an item for the warp's TPW tiles: decode, multiply, add the row sums times
// the unit's factors f (g * 2^-sigma of the lane's two columns).
template <int NT, int TPW, int H>
__device__ __forceinline__ void nv_half(const uint8_t* stage, const uint8_t* bf, const int (&r0)[TPW], int g, int tig,
                                        int lane, const bool (&live)[NT], uint32_t sel0, uint32_t sel1,
                                        const float (&f)[NT][2], float (&acc)[TPW][NT][4]) {
    // B fragments of the half's 8 slices (4 records of 16 bytes per tile)
    uint32_t b[NT][kSlices][2];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
#pragma unroll
        for (int p = 0; p < kSlices / 2; ++p) {
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (live[t]) v = *reinterpret_cast<const uint4*>(bf + t * 4096 + (4 * H + p) * 512 + lane * 16);
            b[t][2 * p][0] = v.x;
            b[t][2 * p][1] = v.y;
            b[t][2 * p + 1][0] = v.z;
            b[t][2 * p + 1][1] = v.w;
        }
    }
#pragma unroll
    for (int tp = 0; tp < TPW; ++tp) {
        // code words c + 4j (swizzled 16-byte chunk 4H + j of the row) and the group scales
        uint32_t w[2][4], sc[2][4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = r0[tp] + 8 * h;  // row % 8 == g
            const uint8_t* cr = stage + row * kCodeRow + tig * 4;
#pragma unroll
            for (int j = 0; j < 4; ++j) w[h][j] = *reinterpret_cast<const uint32_t*>(cr + (((4 * H + j) ^ g) << 4));
            const uint4 s4 = *reinterpret_cast<const uint4*>(stage + kCodeBox + row * kScaleRow);
            // word c + 4j is scale group 8H + 2j + c / 2: byte (2j + c / 2) % 4 of scale word 2H + j / 2
            const uint32_t sw0 = H ? s4.z : s4.x, sw1 = H ? s4.w : s4.y;
            sc[h][0] = e4m3x2_to_f16x2(prmt(sw0, 0u, sel0));
            sc[h][1] = e4m3x2_to_f16x2(prmt(sw0, 0u, sel1));
            sc[h][2] = e4m3x2_to_f16x2(prmt(sw1, 0u, sel0));
            sc[h][3] = e4m3x2_to_f16x2(prmt(sw1, 0u, sel1));
        }
        float c2[2][NT][4];
#define PNQ_NV_SLICE(S)                                                                                       \
    {                                                                                                         \
        constexpr int q = (S) >> 2, bt = (S) & 3;                                                             \
        const uint32_t a0 = hmul2_u32(e2m1x2_to_f16x2<bt>(w[0][2 * q]), sc[0][2 * q]);                        \
        const uint32_t a1 = hmul2_u32(e2m1x2_to_f16x2<bt>(w[1][2 * q]), sc[1][2 * q]);                        \
        const uint32_t a2 = hmul2_u32(e2m1x2_to_f16x2<bt>(w[0][2 * q + 1]), sc[0][2 * q + 1]);                \
        const uint32_t a3 = hmul2_u32(e2m1x2_to_f16x2<bt>(w[1][2 * q + 1]), sc[1][2 * q + 1]);                \
        _Pragma("unroll") for (int t = 0; t < NT; ++t) {                                                      \
            if constexpr ((S) < 2)                                                                            \
                mma_f16_16816_z(c2[(S) & 1][t], a0, a1, a2, a3, b[t][S][0], b[t][S][1]);                      \
            else                                                                                              \
                mma_f16_16816(c2[(S) & 1][t], a0, a1, a2, a3, b[t][S][0], b[t][S][1]);                        \
        }                                                                                                     \
    }
        PNQ_NV_SLICE(0)
        PNQ_NV_SLICE(1)
        PNQ_NV_SLICE(2)
        PNQ_NV_SLICE(3)
        PNQ_NV_SLICE(4)
        PNQ_NV_SLICE(5)
        PNQ_NV_SLICE(6)
        PNQ_NV_SLICE(7)
#undef PNQ_NV_SLICE
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[tp][t][i] = fmaf(c2[0][t][i] + c2[1][t][i], f[t][i & 1], acc[tp][t][i]);
    }
}

template <int NT, int TPW, int H>
__device__ __forceinline__ void nv_consumer_loop(const NvSmem& sm, const Ctx& cx, int i0, int n_items) {
    using C = NvCfg<NT, TPW>;
    const Sched& sc = cx.sc;
    const int M = cx.M, NS = cx.NS, RB = cx.RB, U = sc.U;
    const bool resident = (cx.flags & kResident) != 0;
    const int u0 = sc.unit_of(i0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tig = lane & 3;
    const int tg = warp % C::TG;
    const uint32_t sel0 = (tig >> 1) * 0x11u, sel1 = (2 + (tig >> 1)) * 0x11u;  // scale byte twice
    bool live[NT];  // B column 8t + g holds activation row 8t + g
#pragma unroll
    for (int t = 0; t < NT; ++t) live[t] = (8 * t + g) < M;
    int r0[TPW];
#pragma unroll
    for (int tp = 0; tp < TPW; ++tp) r0[tp] = 16 * (TPW * tg + tp) + g;
    float* part = sm.part();
    bool ok = true;
    float acc[TPW][NT][4];  // [rows g | g + 8][columns 2c | 2c + 1]: c0, c1 row g, c2, c3 row g + 8
#pragma unroll
    for (int tp = 0; tp < TPW; ++tp)
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[tp][t][i] = 0.0f;
    int e = 0;
    auto emit = [&]() {
        const int buf = e & 1;
        if (e >= 2 && !mbar_wait_warp(sm.part_free(buf), ((e >> 1) - 1) & 1)) {
            ok = false;
            return;
        }
#pragma unroll
        for (int tp = 0; tp < TPW; ++tp)
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int m = 8 * t + 2 * tig + i;
                    if (m < M) {
                        float* dst = part + ((H * 2 + buf) * M + m) * kPartPitch + r0[tp];
                        dst[0] = acc[tp][t][i];
                        dst[8] = acc[tp][t][2 + i];
                    }
                    acc[tp][t][i] = acc[tp][t][2 + i] = 0.0f;
                }
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.part_full(buf));
        ++e;
    };
    int t_i = sc.tile_of(i0), u_i = sc.unit_of(i0);
    int cur_t = t_i, r = -1, u_run = -1;
    for (int gi = 0; gi < n_items && ok; ++gi, next_item(sc, t_i, u_i)) {
        if (t_i != cur_t) {
            emit();
            if (!ok) break;
            cur_t = t_i;
        }
        if (!resident && u_i != u_run) {  // a new run: its operands
            if (!consumer_next_run(sm, RB, lane, r)) {
                ok = false;
                break;
            }
            u_run = u_i;
        }
        const int s = gi % NS;
        if (!mbar_wait_warp(sm.full(s), (gi / NS) & 1)) {
            ok = false;
            break;
        }
        const int os = resident ? ((u_i >= u0) ? u_i - u0 : u_i - u0 + U) : r % RB;
        const float* so = sm.slot_so<NT>(os);
        float f[NT][2];  // g * 2^-sigma of the unit for the lane's columns 2c, 2c + 1
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int m = 8 * t + 2 * tig + i;
                f[t][i] = (m < M) ? so[m] : 0.0f;
            }
        nv_half<NT, TPW, H>(sm.stage(s), sm.slot(os), r0, g, tig, lane, live, sel0, sel1, f, acc);
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.empty(s));
    }
    if (ok && n_items > 0) emit();
    if (!ok && lane == 0) record_error(cx.err, kErrFullWait);
}

template <int NT, int TPW>
__global__ void __launch_bounds__(NvCfg<NT, TPW>::THREADS, 1) nvfp4_gemv_kernel(const __grid_constant__ NvArgs a) {
    using C = NvCfg<NT, TPW>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const NvSmem sm{base,       smem_addr(base), a.NS,       a.RB,         a.M,          a.list_off, a.part_off,
                    a.xs_off,   a.ring_off,      a.stage_off, a.slot_bytes, a.list_cap};
    const Ctx cx{a.sc, a.X, a.Y, a.ws, a.cnt, a.err, a.N, a.K, a.M, a.NS, a.RB, a.flags};
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const Sched& sc = cx.sc;
    const int i0 = sc.first(blockIdx.x), i1 = sc.first(blockIdx.x + 1);
    const int n_items = i1 - i0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.NS; ++s) {
            mbar_init(sm.full(s), 1);
            mbar_init(sm.empty(s), C::CW);
        }
        for (int s = 0; s < a.RB; ++s) {
            mbar_init(sm.op_full(s), C::NB);
            mbar_init(sm.op_empty(s), C::CW);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(sm.part_full(b), C::CW);
            mbar_init(sm.part_free(b), 1);
        }
        mbar_init(sm.x_free(), 1);
        mbar_fence_init();
        griddep_launch_dependents();
        *sm.n_finish() = 0;
    }
    __syncthreads();

    if (warp == C::PRODUCER) {
        // ---------------- producer: codes and scales of one item per stage ----------------
        if (lane == 0 && n_items > 0) {
            const uint64_t pol = l2_policy_evict_first();
            bool ok = true;
            int t_n = sc.tile_of(i0), u_n = sc.unit_of(i0);
            const int x_stage = (cx.flags & kXOverlap) ? a.x_stage : cx.NS;  // stages holding x at first
            auto issue = [&](int gi) {
                const int s = gi % cx.NS;
                if (gi >= cx.NS) {
                    if (!mbar_wait_bounded(sm.empty(s), ((gi / cx.NS) - 1) & 1)) return false;
                } else if (s >= x_stage) {
                    if (!mbar_wait_bounded(sm.x_free(), 0)) return false;
                }
                mbar_arrive_expect_tx(sm.full(s), static_cast<uint32_t>(kStageBytes));
                const uint32_t dst = smem_addr(sm.stage(s));
                tma_load_2d(dst, &a.codes_map, u_n * (kCodeRow / 4), t_n * kTileRows, sm.full(s), pol);
                tma_load_2d(dst + kCodeBox, &a.scales_map, u_n * (kScaleRow / 4), t_n * kTileRows, sm.full(s), pol);
                next_item(sc, t_n, u_n);
                return true;
            };
            int gi = 0;
            if (cx.flags & kStaticWeights) {
                // the weights are not written by earlier work in the stream: fill the stages
                // (those not holding x) before the previous grid completes
                for (; ok && gi < min(n_items, min(x_stage, a.pf)); ++gi) ok = issue(gi);
            }
            griddep_wait();  // without the static-weights flag W may be written by the previous grid
            for (; ok && gi < n_items; ++gi) ok = issue(gi);
            if (!ok) record_error(cx.err, kErrEmptyWait);
            // every copy issued has landed before the CTA may exit
            bool drained = true;
            for (int gg = max(0, gi - cx.NS); drained && gg < gi; ++gg)
                drained = mbar_wait_bounded(sm.full(gg % cx.NS), (gg / cx.NS) & 1);
            if (!drained) record_error(cx.err, kErrDrainWait);
        }
        __syncwarp();
    } else if (warp == C::REDUCER) {
        // ---------------- reducer: row sums -> Y or workspace ----------------
        if (n_items > 0) {
            griddep_wait();  // the workspace, the counters and Y belong to earlier grids until now
            bool ok = true;
            int e = 0, np = 0;
            int t_i = sc.tile_of(i0), u_i = sc.unit_of(i0);
            int u_first = u_i, n_run = 0;
            for (int gi = 0; gi < n_items && ok; ++gi) {
                const int t_cur = t_i;
                ++n_run;
                next_item(sc, t_i, u_i);
                if (gi + 1 < n_items && t_i == t_cur) continue;
                const int buf = e & 1;
                if (!mbar_wait_warp(sm.part_full(buf), (e >> 1) & 1)) {
                    ok = false;
                    break;
                }
                if (reduce_share<8 * NT>(cx, sm, buf, t_cur, u_first, n_run, lane)) {
                    if (lane == 0) sm.pending()[np] = t_cur;
                    ++np;
                }
                ++e;
                u_first = u_i;
                n_run = 0;
            }
            if (np > 0) count_shares(cx, sm, np, lane);
            if (!ok && lane == 0) record_error(cx.err, kErrReduceWait);
        }
    } else if (a.flags & kResident) {
        // ---------------- resident operands: consumers and builders build all units' ----------------
        // (unit slot k = unit u0 + k mod U; jobs = (slot, row))
        if (n_items > 0) {
            const int u0 = sc.unit_of(i0);
            const int span = sc.span(i0, i1);
            const int pw = (warp < C::CW) ? warp : warp - C::BUILDER + C::CW;
            const int M = cx.M;
            auto copy = [&](int row) {  // x row slot row = k * M + m, by one warp (32 chunks of 16 bytes)
                const int k = row / M, m = row - k * M;
                int u = u0 + k;
                if (u >= sc.U) u -= sc.U;
                cp_async16(smem_addr(sm.xs(k) + m * kUnitK) + 16u * lane,
                           a.X + static_cast<size_t>(m) * cx.K + static_cast<size_t>(u) * kUnitK + 8 * lane);
            };
            const bool overlap = (a.flags & kXOverlap) != 0;
            auto job = [&](int i) {
                const int k = i / M, m = i - k * M;
                nv_build_row<NT>(sm.slot(k), sm.slot_so<NT>(k), sm.xs(k) + m * kUnitK, m, a.g, lane);
            };
            resident_prologue(pw, C::CW + C::NB, span * M, span * M, overlap, copy, job);
            if (threadIdx.x == 0 && overlap) mbar_arrive(sm.x_free());
            if (warp < C::TG)
                nv_consumer_loop<NT, TPW, 0>(sm, cx, i0, n_items);
            else if (warp < C::CW)
                nv_consumer_loop<NT, TPW, 1>(sm, cx, i0, n_items);
        }
    } else if (warp >= C::BUILDER) {
        // ---------------- builders: operands of each run; rows m = b, b + NB, .. ----------------
        if (n_items > 0) {
            griddep_wait();  // X belongs to the previous grid until now
            const int b = warp - C::BUILDER;
            auto issue = [&](int u, int buf) {
                uint16_t* xb = sm.xs(buf);
                for (int m = b; m < cx.M; m += C::NB)
                    cp_async16(smem_addr(xb + m * kUnitK) + 16u * lane,
                               a.X + static_cast<size_t>(m) * cx.K + static_cast<size_t>(u) * kUnitK + 8 * lane);
            };
            auto build = [&](int slot, int buf) {
                const uint16_t* xb = sm.xs(buf);
                for (int m = b; m < cx.M; m += C::NB)
                    nv_build_row<NT>(sm.slot(slot), sm.slot_so<NT>(slot), xb + m * kUnitK, m, a.g, lane);
            };
            bool ok;
            if (a.XB == 4)
                ok = builder_loop<4>(sm, sc, i0, n_items, cx.RB, lane, issue, build);
            else if (a.XB == 2)
                ok = builder_loop<2>(sm, sc, i0, n_items, cx.RB, lane, issue, build);
            else
                ok = builder_loop<1>(sm, sc, i0, n_items, cx.RB, lane, issue, build);
            if (!ok && lane == 0) record_error(cx.err, kErrOperandWait);
        }
    } else {
        // ---------------- consumer warps ----------------
        if (n_items > 0) {
            if (warp < C::TG)
                nv_consumer_loop<NT, TPW, 0>(sm, cx, i0, n_items);
            else
                nv_consumer_loop<NT, TPW, 1>(sm, cx, i0, n_items);
        }
    }
    // the tiles this CTA completed: every warp sums some of them
    __syncthreads();
    finish_tiles(cx, sm, warp, C::THREADS / 32, lane);
}

// ---- host side --------------------------------------------------------------------------------------

constexpr int kDefaultStages = 8;

struct NvPlan {
    Sched sc{};
    bool publish = false;
    unsigned mode = 0;  // kResident, kXOverlap
    int NS = 0, RB = 0, XB = 0, x_stage = 0, list_cap = 0;
    uint32_t list_off = 0, part_off = 0, xs_off = 0, ring_off = 0, stage_off = 0, slot_bytes = 0, total = 0;
};

// Barriers, lists and row sums at the start; returns the first free (128-aligned) offset.
uint32_t nv_head_layout(int bfu, int M, int NS, int RB, NvPlan& p) {
    p.list_cap = (p.sc.items + p.sc.G - 1) / p.sc.G;
    p.list_off = align_up(8u * (2u * NS + 2u * RB + 5u), 16);  // full, empty, op_full, op_empty, part x 4, x_free
    p.part_off = align_up(p.list_off + (2u * p.list_cap + 4u) * 4u, 16);
    p.slot_bytes = align_up(static_cast<uint32_t>(bfu) + 64u, 128);
    return align_up(p.part_off + 4u * M * kPartPitch * 4u, 128);
}

bool nv_layout(int bfu, int M, int NS, int RB, int XB, NvPlan& p) {
    p.xs_off = nv_head_layout(bfu, M, NS, RB, p);
    p.ring_off = align_up(p.xs_off + static_cast<uint32_t>(XB) * M * kUnitK * 2u, 128);
    p.stage_off = align_up(p.ring_off + static_cast<uint32_t>(RB) * p.slot_bytes, 1024);
    const uint64_t total = p.stage_off + static_cast<uint64_t>(NS) * kStageBytes;
    if (total + 1024u > kSmemLimit) return false;
    p.mode = 0;
    p.NS = NS;
    p.RB = RB;
    p.XB = XB;
    p.total = static_cast<uint32_t>(total);
    return true;
}

// Resident layout: one operand slot per unit of the largest share, x of the share in its own
// region or (overlap) in the last weight stages until the operands are built.
bool nv_layout_resident(int bfu, int M, int NS, bool overlap, NvPlan& p) {
    int span = 0;
    for (int c = 0; c < p.sc.G; ++c) span = std::max(span, p.sc.span(p.sc.first(c), p.sc.first(c + 1)));
    uint64_t off = nv_head_layout(bfu, M, NS, 0, p);
    const uint64_t xbytes = static_cast<uint64_t>(span) * M * kUnitK * 2u;
    if (!overlap) {
        p.xs_off = static_cast<uint32_t>(off);
        off = (off + xbytes + 127) / 128 * 128;
    }
    p.ring_off = static_cast<uint32_t>(off);
    const uint64_t stage_off = (off + static_cast<uint64_t>(span) * p.slot_bytes + 1023) / 1024 * 1024;
    const uint64_t total = stage_off + static_cast<uint64_t>(NS) * kStageBytes;
    if (total + 1024u > kSmemLimit) return false;
    p.stage_off = static_cast<uint32_t>(stage_off);
    p.x_stage = NS;
    if (overlap) {
        const int x_stages = static_cast<int>((xbytes + kStageBytes - 1) / kStageBytes);
        if (x_stages > NS) return false;
        p.x_stage = NS - x_stages;
        p.xs_off = p.stage_off + static_cast<uint32_t>(p.x_stage) * kStageBytes;
    }
    p.mode = kResident | (overlap ? kXOverlap : 0u);
    p.NS = NS;
    p.RB = 0;
    p.XB = 0;
    p.total = static_cast<uint32_t>(total);
    return true;
}

bool nv_fit_resident(int bfu, int M, int ns_req, NvPlan& p) {
    const int ns_max = ns_req > 0 ? ns_req : kDefaultStages, ns_lo = ns_req > 0 ? ns_req : 3;
    for (bool overlap : {false, true})
        for (int ns = ns_max; ns >= ns_lo; --ns)
            if (nv_layout_resident(bfu, M, ns, overlap, p)) return true;
    return false;
}

bool nv_fit_stream(int bfu, int M, int ns_req, int rb_req, NvPlan& p) {
    const int ns_max = ns_req > 0 ? ns_req : kDefaultStages;
    for (int ns_min : {3, 2})
        for (int xb : {4, 2, 1})
            for (int rb : {3, 2}) {
                if (rb_req > 0 && rb != 3) continue;
                const int r = rb_req > 0 ? std::min(std::max(rb_req, 2), 4) : rb;  // one slot would deadlock
                for (int ns = ns_max; ns >= (ns_req > 0 ? ns_req : ns_min); --ns)
                    if (nv_layout(bfu, M, ns, r, xb, p)) return true;
            }
    return false;
}

// The PN path's choice: tile-major items with resident operands when they fit (stream-K grid
// or one CTA per tile); otherwise, for wide batches, tile-major items with the streaming ring
// (order = 2: grouped unit-major items with resident operands when they fit).
bool nv_plan(int bfu, int M, int64_t T, int64_t U, int sms, bool grid_forced, int ns_req, int rb_req, int order,
             NvPlan& p) {
    const int64_t items = T * U;
    const int64_t G0 = std::min<int64_t>(sms, items);
    int64_t cands[2] = {G0, 0};
    if (!grid_forced && T < sms) cands[1] = T;
    auto base = [&](int64_t G) {
        NvPlan q;
        q.sc.items = static_cast<int>(items);
        q.sc.T = static_cast<int>(T);
        q.sc.U = static_cast<int>(U);
        q.sc.G = static_cast<int>(G);
        q.sc.tile_major = 1;
        q.sc.tg = 1;
        return q;
    };
    auto publishes = [](const NvPlan& q) {
        if (!q.sc.tile_major && q.sc.U > 1) return true;
        for (int c = 1; c < q.sc.G; ++c)
            if (q.sc.tile_of(q.sc.first(c)) == q.sc.tile_of(q.sc.first(c) - 1)) return true;
        return false;
    };
    bool found = false;
    double best = 0.0;
    if (rb_req <= 0 && order != 2)
        for (int64_t G : cands) {
            if (G <= 0) continue;
            NvPlan q = base(G);
            if (!nv_fit_resident(bfu, M, ns_req, q)) continue;
            q.publish = publishes(q);
            // items here are half the bytes of a PN item: the reduction tail weighs more
            const double cost = static_cast<double>((items + G - 1) / G) + (q.publish ? 5.0 : 0.0);
            if (!found || cost < best) {
                best = cost;
                p = q;
                found = true;
            }
        }
    if (found) return true;
    if (rb_req <= 0 && order == 2 && T > 1 && U > 1) {
        for (int64_t tg : {2, 4, 8, 16, 32, 64, 128}) {
            NvPlan q = base(G0);
            q.sc.tile_major = 0;
            q.sc.tg = static_cast<int>(std::min<int64_t>(tg, T));
            if (nv_fit_resident(bfu, M, ns_req, q)) {
                q.publish = publishes(q);
                p = q;
                return true;
            }
            if (tg >= T) break;
        }
    }
    NvPlan q = base(G0);
    if (!nv_fit_stream(bfu, M, ns_req, rb_req, q)) return false;
    q.publish = publishes(q);
    p = q;
    return true;
}

// Environment override PNQ_NV_CFG="tpw,grid,rb,ns,order,pf" (fields 0 = automatic), read once.
MmaConfig nv_env_config() {
    static MmaConfig cfg = [] {
        MmaConfig c{0, 0, 0, 0, 0, 0};
        if (const char* s = std::getenv("PNQ_NV_CFG")) {
            int v[6] = {0, 0, 0, 0, 0, 0};
            int n = 0;
            const char* p = s;
            while (*p && n < 6) {
                v[n++] = static_cast<int>(std::strtol(p, const_cast<char**>(&p), 10));
                if (*p == ',') ++p;
            }
            c = MmaConfig{v[0], v[1], v[2], v[3], v[4], v[5]};
        }
        return c;
    }();
    return cfg;
}

template <int NT, int TPW>
cudaError_t nv_launch_cfg(NvArgs& a, const MmaConfig& cfg, bool static_weights, cudaStream_t stream,
                          const ExtWorkspace& ext) {
    using C = NvCfg<NT, TPW>;
    NvPlan p;
    const int cap = cfg.grid > 0 ? std::min(cfg.grid, device_sm_count()) : device_sm_count();
    if (!nv_plan(C::BFU, a.M, a.sc.T, a.sc.U, cap, cfg.grid > 0, cfg.ns, cfg.rb, cfg.order, p))
        return cudaErrorNotSupported;
    auto kern = nvfp4_gemv_kernel<NT, TPW>;
    static std::atomic<bool> opted[64];  // the attribute is set once per device (threads may race to set it)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!opted[dev].load(std::memory_order_relaxed)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemLimit));
        if (e != cudaSuccess) return e;
        opted[dev].store(true, std::memory_order_relaxed);
    }
    const size_t ws_floats = static_cast<size_t>(a.sc.T) * a.sc.U * a.M * kTileRows;
    if (ext.ws) {
        if (p.publish && (ext.floats < ws_floats || ext.counters < static_cast<size_t>(a.sc.T)))
            return cudaErrorMemoryAllocation;
        a.ws = ext.ws;
        a.cnt = ext.cnt;
    } else {
        e = stream_workspace(stream, ws_floats, static_cast<size_t>(a.sc.T), &a.ws, &a.cnt);
        if (e != cudaSuccess) return e;
    }
    a.sc = p.sc;
    a.NS = p.NS;
    a.RB = p.RB;
    a.XB = p.XB;
    a.flags = (static_weights ? kStaticWeights : 0u) | p.mode;
    a.x_stage = p.x_stage;
    a.pf = cfg.pf > 0 ? cfg.pf : p.NS;
    a.list_off = p.list_off;
    a.list_cap = p.list_cap;
    a.part_off = p.part_off;
    a.xs_off = p.xs_off;
    a.ring_off = p.ring_off;
    a.stage_off = p.stage_off;
    a.slot_bytes = p.slot_bytes;
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(p.sc.G, 1, 1);
    lc.blockDim = dim3(C::THREADS, 1, 1);
    lc.dynamicSmemBytes = p.total + 1024u;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, kern, a);
}

}  // namespace

cudaError_t launch_nvfp4_gemv_mma(const Nvfp4View& w, int64_t N, int64_t K, const uint16_t* X, int M, float* Y,
                                  int* err, MmaConfig cfg, bool static_weights, cudaStream_t stream,
                                  const ExtWorkspace& ext) {
    if (N == 0) return cudaSuccess;
    if (K % kUnitK != 0 || M < 1 || M > 16) return cudaErrorNotSupported;
    const int64_t U = K / kUnitK, T = (N + kTileRows - 1) / kTileRows;
    if (N > INT32_MAX || K > INT32_MAX || T * U > INT32_MAX) return cudaErrorNotSupported;
    if (reinterpret_cast<uintptr_t>(w.codes) % 16 != 0 || reinterpret_cast<uintptr_t>(w.scales) % 16 != 0 ||
        reinterpret_cast<uintptr_t>(X) % 16 != 0)
        return cudaErrorNotSupported;
    NvArgs a{};
    if (!encode_u32_map(&a.codes_map, w.codes, N, K / 8, kCodeRow / 4, kTileRows, true) ||
        !encode_u32_map(&a.scales_map, w.scales, N, K / 64, kScaleRow / 4, kTileRows, false))
        return cudaErrorNotSupported;
    a.X = X;
    a.Y = Y;
    a.err = err;
    a.g = w.g;
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.M = M;
    a.sc.T = static_cast<int>(T);
    a.sc.U = static_cast<int>(U);
    a.sc.items = static_cast<int>(T * U);
    const MmaConfig env = nv_env_config();
    if (cfg.tpw <= 0) cfg.tpw = env.tpw;
    if (cfg.grid <= 0) cfg.grid = env.grid;
    if (cfg.rb <= 0) cfg.rb = env.rb;
    if (cfg.ns <= 0) cfg.ns = env.ns;
    if (cfg.order <= 0) cfg.order = env.order;
    if (cfg.pf <= 0) cfg.pf = env.pf;
    const int nt = (M + 7) / 8;
    // two row tiles per consumer warp (8 consumer warps, each scale and B fragment load serving
    // two tiles) measured faster than one at every M (17408 x 5120, M = 1: 22.5 vs 24.5 us)
    const int tpw = cfg.tpw > 0 ? cfg.tpw : 2;
    if (nt == 1) return tpw == 1 ? nv_launch_cfg<1, 1>(a, cfg, static_weights, stream, ext)
                                 : nv_launch_cfg<1, 2>(a, cfg, static_weights, stream, ext);
    return tpw == 1 ? nv_launch_cfg<2, 1>(a, cfg, static_weights, stream, ext)
                    : nv_launch_cfg<2, 2>(a, cfg, static_weights, stream, ext);
}

}  // namespace pnq
