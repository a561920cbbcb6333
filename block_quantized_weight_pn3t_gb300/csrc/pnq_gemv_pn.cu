// pnq_gemv_pn.cu -- PN (pn3t / pn4t) GEMV on the tensor cores with mma.sync, sm_103a (fast path).
//
// Computes Y[m][n] = sum_k w[n][k] x[m][k] for 1 <= M <= 16, with w = d * (n - z) decoded in
// registers from the 34-byte blocks of the "PN weight format" page (sections Block layout and
// Value) just before the multiply.
//
// Why mma.sync. A GEMV streams every weight once; at HBM rate an SM has to take in about 50
// weights per cycle. The warp-level m16n8k16 MMA sustains 0.5 instructions per cycle per SM
// (256 weights each), while a tcgen05.mma of M = 128, K = 16 occupies the tensor core for about
// 100 cycles whatever N <= 128 is (2048 weights each) -- both measured on this part -- so for
// the narrow N of a GEMV the warp-level MMA has the throughput and tcgen05 does not.
//
// Items and schedule (stream-K, pnq_streamk.cuh). The weight matrix is cut into items of 128
// rows x one K unit of 8 blocks (272 bytes per row), numbered tile-major (grouped unit-major for
// wide batches whose operands would not fit otherwise); every CTA of a persistent grid (one per
// SM) takes an equal contiguous share, so all SMs stream the same number of bytes.
//
// Memory pipeline. One producer thread loads one item per stage with a 2-D tensor-map copy
// (box 272 bytes x 128 rows, L2 evict-first; rows past N read as zeros) into an NS-stage ring
// under mbarriers. With the static-weights flag the first stages are requested before the
// previous grid in the stream has finished.
//
// Decode and multiply (consumer warps). Warp = TPW tiles of 16 rows x half a unit (4 blocks).
// A 32-bit word of a block holds two codes at the same shift in its two 16-bit halves; masking
// out one such pair leaves in each half the exact fp16 subnormal n * 2^-24 * 8^j (pn3t; 16^j
// for pn4t, j = position of the pair): one AND per two weights gives an mma A register. Lane
// (g, c) of the warp uses words c and c + 4 of rows g and g + 8; the k order inside a block is
// free as long as B uses the same order, so the 2-byte aligned words of even blocks are read as
// aligned words pairing the high half of word i-1 with the low half of word i (one PRMT).
//
// B operand: x times 8^-j (16^-j) times 2^sigma (per K unit and activation row, so that
// max|x| * 2^sigma lies in [2^14, 2^15)), split into fp16 hi + lo parts (~21 bits: hi = the
// leading 11 bits by truncation, lo = the rest rounded to fp16) that take mma columns 2m and
// 2m + 1 (NT = ceil(2M / 8) n8 tiles), stored per block in register order. Beside them:
// Z = z * 2^(sigma - 24) * (sum of the block's x), and 2^(24 - sigma). Built once per K unit of
// the CTA's share by all consumer and builder warps before the first item (resident mode), or,
// when those operands do not fit, by the builder warps into a ring ahead of the consumers.
//
// Block scale and zero point: per item a_m = sum over its blocks of d * (c - Z); the tile's row
// sum gains a_m * 2^(24 - sigma).
//
// Reduction (pnq_streamk.cuh): whole tiles go from the reducer warp to Y, shares of a tile
// that several CTAs cover meet in the workspace and are summed in unit order.
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

constexpr int kUnitBlocks = 8;                         // blocks per K unit
constexpr int kUnitBytes = kUnitBlocks * kBlockBytes;  // 272 bytes of a row per unit
constexpr int kUnitU32 = kUnitBytes / 4;               // 68
constexpr int kStageBytes = kTileRows * kUnitBytes;    // 34816
constexpr int kHalfBlocks = 4;                         // blocks per consumer warp and item

template <int TYPE, int NT, int TPW>
struct Cfg {
    static constexpr int STEPS = PnFmt<TYPE>::PAIRS;
    static constexpr int UK = kUnitBlocks * PnFmt<TYPE>::BLK;  // weights of a row per unit
    static constexpr int TG = 8 / TPW;             // tile groups per half
    static constexpr int CW = 2 * TG;              // consumer warps
    static constexpr int NB = (TPW == 1 || NT >= 4) ? 2 : 6;  // builder warps (within the register budget)
    static constexpr int PRODUCER = CW, REDUCER = CW + 1, BUILDER = CW + 2;
    static constexpr int THREADS = 32 * (CW + 2 + NB);
    // B records: per block, n8 tile and pair of slices a group of `lg` 16-byte lane records; all
    // 32 lanes with several tiles, only the lanes of columns < 2M (lg = 8M) with one
    static __host__ __device__ int lg(int M) { return NT == 1 ? (8 * M < 32 ? 8 * M : 32) : 32; }
    static __host__ __device__ int bfu(int M) { return NT * STEPS * lg(M) * 8; }  // bytes per block
};

struct PnArgs {
    CUtensorMap map;  // weights as u32 [N][row_bytes / 4], box {68, 128}
    const float* X;
    float* Y;
    float* ws;       // partial rows [T][U][M][128]: slot (t, u) = the share of tile t starting at unit u
    uint32_t* cnt;   // [T] shares counted per row tile (zero between launches)
    int* err;
    Sched sc;
    int N, K, M, NS, RB, XB;
    int x_stage;     // resident mode with x in the weight stages: the first stage holding x
    int pf;          // static weights: stages requested before griddepcontrol.wait
    unsigned flags;  // kStaticWeights, kResident, kXOverlap
    uint32_t list_off, part_off, xs_off, ring_off, stage_off, slot_bytes;
    int list_cap;
};

// 2^-(BITS * jj) for slice j, and its inverse.
template <int TYPE>
__device__ __forceinline__ float step_scale(int j) {
    return (TYPE == kTypePn3t) ? ((j % 3 == 0) ? 1.0f : (j % 3 == 1) ? 0.125f : 0.015625f)
                               : ((j & 1) ? 0.0625f : 1.0f);
}
template <int TYPE>
__device__ __forceinline__ float step_scale_inv(int j) {
    return (TYPE == kTypePn3t) ? ((j % 3 == 0) ? 1.0f : (j % 3 == 1) ? 8.0f : 64.0f) : ((j & 1) ? 16.0f : 1.0f);
}

// Masked pair J of a word (w) or of the word shifted right by 9 (pn3t) / 8 (pn4t) (s).
template <int TYPE, int J>
__device__ __forceinline__ uint32_t code_pair(uint32_t w, uint32_t s) {
    if constexpr (TYPE == kTypePn3t) {
        if constexpr (J < 3) return w & (0x00070007u << (3 * J));
        else return s & (0x00070007u << (3 * (J - 3)));
    } else {
        if constexpr (J < 2) return w & (0x000F000Fu << (4 * J));
        else return s & (0x000F000Fu << (4 * (J - 2)));
    }
}

// Element (within a block) that the low (hi_half = 0) or high half of decode register i holds
// for pair j. Odd blocks start 2 bytes past a 4-byte boundary: register i is word i. Even
// blocks: register i (i >= 1) is the aligned word at byte 4i = high half of word i-1 and low
// half of word i; register 0 pairs the low half of word 0 with the high half of word 7.
__device__ __forceinline__ int pn_elem(int cpw, int odd_block, int i, int j, int hi_half) {
    if (odd_block) return cpw * i + 2 * j + hi_half;
    if (i == 0) return hi_half ? cpw * 7 + 2 * j + 1 : 2 * j;
    return hi_half ? cpw * i + 2 * j : cpw * (i - 1) + 2 * j + 1;
}

__device__ __forceinline__ uint32_t lds32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }
__device__ __forceinline__ float ld_half(const uint8_t* p) {
    return __half2float(*reinterpret_cast<const __half*>(p));
}

// Shared-memory regions (offsets from the 1024-aligned base): barriers at 0, lists, row sums,
// x buffers, operand slots (a ring, or one per unit of the share in resident mode), weight
// stages. Resident mode keeps x as [unit slot][M][UK] (possibly inside the last weight stages).
struct Smem {
    uint8_t* base;
    uint32_t bar0;  // shared address of barrier 0
    int NS, RB, M, UK;
    uint32_t list_off, part_off, xs_off, ring_off, stage_off, slot_bytes, z_off;
    int list_cap;
    __device__ uint32_t full(int s) const { return bar0 + 8u * s; }
    __device__ uint32_t empty(int s) const { return bar0 + 8u * (NS + s); }
    __device__ uint32_t op_full(int s) const { return bar0 + 8u * (2 * NS + s); }
    __device__ uint32_t op_empty(int s) const { return bar0 + 8u * (2 * NS + RB + s); }
    __device__ uint32_t part_full(int b) const { return bar0 + 8u * (2 * NS + 2 * RB + b); }
    __device__ uint32_t part_free(int b) const { return bar0 + 8u * (2 * NS + 2 * RB + 2 + b); }
    __device__ uint32_t x_free() const { return bar0 + 8u * (2 * NS + 2 * RB + 4); }
    __device__ float* part() const { return reinterpret_cast<float*>(base + part_off); }
    int J;  // builder jobs per run (x rows per buffer)
    __device__ float* xs(int buf) const {  // [J][UK] x rows of one K unit, one per builder job
        return reinterpret_cast<float*>(base + xs_off) + static_cast<size_t>(buf) * J * UK;
    }
    __device__ uint8_t* slot(int s) const { return base + ring_off + static_cast<uint32_t>(s) * slot_bytes; }
    __device__ float* slot_z(int s) const { return reinterpret_cast<float*>(slot(s) + z_off); }  // [8][M]
    __device__ float* slot_so(int s) const { return slot_z(s) + kUnitBlocks * M; }                // [M]
    __device__ uint8_t* stage(int s) const { return base + stage_off + static_cast<uint32_t>(s) * kStageBytes; }
    // tiles whose partial shares wait to be counted, tiles this CTA completes (list_cap entries
    // each, list_cap >= the items of any CTA), and the number of the latter
    __device__ int* n_finish() const { return reinterpret_cast<int*>(base + list_off); }
    __device__ int* pending() const { return reinterpret_cast<int*>(base + list_off) + 4; }
    __device__ int* finish() const { return reinterpret_cast<int*>(base + list_off) + 4 + list_cap; }
};

// B fragments of one block for every n8 tile: lanes whose column is in use load their records,
// the others hold zeros. rs = bytes of a record group (lg * 16).
template <int TYPE, int NT>
__device__ __forceinline__ void load_bfrag(const uint8_t* bf, int lane, const bool (&live)[NT], int rs,
                                           uint32_t (&b)[NT][PnFmt<TYPE>::PAIRS][2]) {
    constexpr int STEPS = PnFmt<TYPE>::PAIRS;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const uint8_t* base = bf + t * (rs / 2) * STEPS;
#pragma unroll
        for (int q = 0; q < STEPS / 2; ++q) {
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (live[t]) v = *reinterpret_cast<const uint4*>(base + q * rs + lane * 16);
            b[t][2 * q][0] = v.x;
            b[t][2 * q][1] = v.y;
            b[t][2 * q + 1][0] = v.z;
            b[t][2 * q + 1][1] = v.w;
        }
        if constexpr (STEPS & 1) {
            uint2 v = make_uint2(0u, 0u);
            if (live[t]) v = *reinterpret_cast<const uint2*>(base + (STEPS / 2) * rs + lane * 8);
            b[t][STEPS - 1][0] = v.x;
            b[t][STEPS - 1][1] = v.y;
        }
    }
}

// Per-lane constants of build_row, the same for every block pair, unit and row: the lane builds
// the record of lane column c and record pair pr (slices 2pr, 2pr + 1; registers b0 = decode
// register c, b1 = register c + 4) for blocks of parity `odd` (JL lanes per block, blocks of a
// pass start at an even index). off[q][h] = element of half h of register q, ss[q] = step scale.
template <int TYPE>
struct BuildLane {
    static constexpr int STEPS = PnFmt<TYPE>::PAIRS;
    static constexpr int PAIRS = (STEPS + 1) / 2;           // records per lane column and block
    static constexpr int JL = (PAIRS * 4 <= 8) ? 8 : 16;    // lanes per block
    static constexpr int BPP = 32 / JL;                     // blocks per pass
    int off[4][2];
    float ss[4];
    int pr, c;
    unsigned act;  // bit q: slice 2pr + q / 2 exists
    __device__ explicit BuildLane(int lane) {
        using F = PnFmt<TYPE>;
        const int jl = lane % JL, odd = (lane / JL) & 1;
        pr = jl >> 2;
        c = jl & 3;
        act = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // q = 2 * (slice - 2pr) + register
            const int st = 2 * pr + (q >> 1), i = c + 4 * (q & 1);
            const bool on = pr < PAIRS && st < STEPS;
            act |= on ? (1u << q) : 0u;
            off[q][0] = on ? pn_elem(F::CPW, odd, i, st, 0) : 0;
            off[q][1] = on ? pn_elem(F::CPW, odd, i, st, 1) : 0;
            ss[q] = on ? step_scale<TYPE>(st) : 0.0f;
        }
    }
};

// Operands of activation row m for one K unit, blocks blk0 .. blk0 + NBLK - 1 (one warp): sigma
// from the row's largest |x| over the unit, the blocks' B fragments (hi column 2m, lo column
// 2m + 1; 16-byte lane records, 8-byte for an odd last slice alone; lane = 4 * (column % 8) + c)
// and zero-point terms Z, and (blk0 = 0) 2^(24 - sigma). xr = the row's UK x values in shared
// memory.
template <int TYPE, int NT, int NBLK>
__device__ __forceinline__ void build_row(uint8_t* slot_b, float* slot_z, float* slot_so, const float* xr, int m,
                                          int M, int blk0, int lane, const BuildLane<TYPE>& L, int rs) {
    using F = PnFmt<TYPE>;
    using BL = BuildLane<TYPE>;
    constexpr int STEPS = F::PAIRS;
    constexpr int UK = kUnitBlocks * F::BLK;
    const int ts = (rs / 2) * STEPS, bfu = NT * ts;  // bytes per n8 tile and per block
    uint32_t mx = 0;  // a non-negative float's bits order like its value
#pragma unroll
    for (int q = lane; q < UK / 4; q += 32) {
        const float4 v = reinterpret_cast<const float4*>(xr)[q];
        mx = max(mx, max(max(__float_as_uint(v.x) & 0x7FFFFFFFu, __float_as_uint(v.y) & 0x7FFFFFFFu),
                         max(__float_as_uint(v.z) & 0x7FFFFFFFu, __float_as_uint(v.w) & 0x7FFFFFFFu)));
    }
    mx = __reduce_max_sync(0xffffffffu, mx);
    const int E = static_cast<int>(mx >> 23);
    int sg = (mx == 0 || E >= 255) ? 0 : 141 - E;  // max < 2^(E-126)
    sg = min(100, max(-100, sg));
    const float sig_in = exp2i(sg);
    float sc[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) sc[q] = sig_in * L.ss[q];
    const int n = 2 * m;
    const int lh = ((n & 7) << 2) | L.c, ll = (((n + 1) & 7) << 2) | L.c;
    const bool single = (STEPS & 1) && L.pr == BL::PAIRS - 1;  // the odd last slice alone
    const int jl = lane % BL::JL;
#pragma unroll
    for (int b0 = 0; b0 < NBLK; b0 += BL::BPP) {
        const int blk = blk0 + b0 + lane / BL::JL;
        const float* xb = xr + blk * F::BLK;
        uint64_t zs2 = 0;  // this lane's part of the block's sum of x (each element once), two lanes
        if (L.act) {
            uint32_t hi[4] = {0u, 0u, 0u, 0u}, lo[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (L.act & (1u << q)) {
                    const uint64_t xp = f32x2_pack(xb[L.off[q][0]], xb[L.off[q][1]]);
                    zs2 = f32x2_add(zs2, xp);
                    uint64_t hp, lp;
                    split11x2(f32x2_mul(xp, f32x2_pack(sc[q], sc[q])), hp, lp);
                    float h0, h1, l0, l1;
                    f32x2_unpack(hp, h0, h1);
                    f32x2_unpack(lp, l0, l1);
                    hi[q] = f32x2_to_f16x2(h0, h1);  // exact
                    lo[q] = f32x2_to_f16x2(l0, l1);
                }
            }
            uint8_t* tb = slot_b + blk * bfu + (n >> 3) * ts + L.pr * rs;
            if (single) {
                *reinterpret_cast<uint2*>(tb + lh * 8) = make_uint2(hi[0], hi[1]);
                *reinterpret_cast<uint2*>(tb + ll * 8) = make_uint2(lo[0], lo[1]);
            } else {
                *reinterpret_cast<uint4*>(tb + lh * 16) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(tb + ll * 16) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
        }
        float zs, zs_hi;
        f32x2_unpack(zs2, zs, zs_hi);
        zs += zs_hi;
#pragma unroll
        for (int o = BL::JL / 2; o > 0; o >>= 1) zs += __shfl_xor_sync(0xffffffffu, zs, o);  // within the group
        // Z = z * sum over the block of 2^-24 * 8^j * B = z * 2^(sigma - 24) * (sum of x)
        if (jl == 0) slot_z[blk * M + m] = static_cast<float>(F::Z) * zs * exp2i(sg - 24);
    }
    if (lane == 0 && blk0 == 0) slot_so[m] = exp2i(24 - sg);  // undoes sigma and the 2^-24 of the codes
}

// One block B (of the unit, compile time) for the warp's TPW tiles: decode, multiply, fold
// d * (c - Z) into acc[tile][t][row half] (the item's sums, before 2^(24 - sigma)).
template <int TYPE, int NT, int TPW, int B>
__device__ __forceinline__ void pn_block(const uint8_t* const (&row0)[TPW], int tig, uint32_t sel,
                                         const uint8_t* bf, int lane, const bool (&live)[NT], int rs, const float* zb,
                                         int M, float (&acc)[TPW][NT][2]) {
    using F = PnFmt<TYPE>;
    constexpr int STEPS = F::PAIRS;
    constexpr int OFF = kBlockBytes * B;
    constexpr int SH = (TYPE == kTypePn3t) ? 9 : 8;
    // B fragments (columns past 2M are zero and are not read)
    uint32_t b[NT][STEPS][2];
    load_bfrag<TYPE, NT>(bf, lane, live, rs, b);
    float zt[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const int m = 4 * t + tig;
        zt[t] = (m < M) ? zb[m] : 0.0f;
    }
#pragma unroll
    for (int tp = 0; tp < TPW; ++tp) {
        // rows g (h = 0) and g + 8 (h = 1): decode registers c and c + 4, block scale
        uint32_t ra[2], rb[2];
        float d[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint8_t* rp = row0[tp] + h * 8 * kUnitBytes + OFF;
            if constexpr ((B & 1) == 0) {
                ra[h] = prmt(lds32(rp + 4 * tig), lds32(rp + 32), sel);
                rb[h] = lds32(rp + 16 + 4 * tig);
            } else {
                ra[h] = lds32(rp + 2 + 4 * tig);
                rb[h] = lds32(rp + 18 + 4 * tig);
            }
            d[h] = ld_half(rp);
        }
        const uint32_t sa0 = ra[0] >> SH, sa1 = ra[1] >> SH, sb0 = rb[0] >> SH, sb1 = rb[1] >> SH;
        float c[NT][4];
#define PNQ_SLICE(J)                                                                                         \
    if constexpr (J < STEPS) {                                                                               \
        const uint32_t a0 = code_pair<TYPE, J>(ra[0], sa0), a1 = code_pair<TYPE, J>(ra[1], sa1);             \
        const uint32_t a2 = code_pair<TYPE, J>(rb[0], sb0), a3 = code_pair<TYPE, J>(rb[1], sb1);             \
        _Pragma("unroll") for (int t = 0; t < NT; ++t) {                                                     \
            if constexpr (J == 0)                                                                            \
                mma_f16_16816_z(c[t], a0, a1, a2, a3, b[t][J][0], b[t][J][1]);                               \
            else                                                                                             \
                mma_f16_16816(c[t], a0, a1, a2, a3, b[t][J][0], b[t][J][1]);                                 \
        }                                                                                                    \
    }
        PNQ_SLICE(0)
        PNQ_SLICE(1)
        PNQ_SLICE(2)
        PNQ_SLICE(3)
        PNQ_SLICE(4)
#undef PNQ_SLICE
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            acc[tp][t][0] = fmaf(d[0], (c[t][0] + c[t][1]) - zt[t], acc[tp][t][0]);
            acc[tp][t][1] = fmaf(d[1], (c[t][2] + c[t][3]) - zt[t], acc[tp][t][1]);
        }
    }
}

template <int TYPE, int NT, int TPW, int H>
__device__ __forceinline__ void consumer_loop(const Smem& sm, const Ctx& cx, int i0, int n_items) {
    using C = Cfg<TYPE, NT, TPW>;
    const Sched& sc = cx.sc;
    const int M = cx.M, NS = cx.NS, RB = cx.RB, U = sc.U;
    const bool resident = (cx.flags & kResident) != 0;
    const int u0 = sc.unit_of(i0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tig = lane & 3;
    const int tg = warp % C::TG;  // tile group: rows 16 * TPW * tg ..
    const uint32_t sel = (tig == 0) ? 0x5432u : 0x3210u;  // even blocks: register 0 pairs words 0 and 7
    const int rs = C::lg(M) * 16, bfu = C::bfu(M);  // record group and block fragment bytes
    bool live[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) live[t] = (8 * t + g) < 2 * M;
    float* part = sm.part();
    bool ok = true;
    float acc[TPW][NT][2];
#pragma unroll
    for (int tp = 0; tp < TPW; ++tp)
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[tp][t][0] = acc[tp][t][1] = 0.0f;
    int e = 0;  // row sums handed to the reducer so far
    // hand the row sums of the tile just finished to the reducer, then clear them
    auto emit = [&]() {
        const int buf = e & 1;
        if (e >= 2 && !mbar_wait_warp(sm.part_free(buf), ((e >> 1) - 1) & 1)) {
            ok = false;
            return;
        }
#pragma unroll
        for (int tp = 0; tp < TPW; ++tp)
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const int m = 4 * t + tig;
                if (m < M) {
                    float* dst = part + ((H * 2 + buf) * M + m) * kPartPitch + 16 * (TPW * tg + tp) + g;
                    dst[0] = acc[tp][t][0];
                    dst[8] = acc[tp][t][1];
                }
                acc[tp][t][0] = acc[tp][t][1] = 0.0f;
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
        const uint8_t* stage = sm.stage(s);
        const uint8_t* row0[TPW];
#pragma unroll
        for (int tp = 0; tp < TPW; ++tp) row0[tp] = stage + (16 * (TPW * tg + tp) + g) * kUnitBytes;
        const int os = resident ? ((u_i >= u0) ? u_i - u0 : u_i - u0 + U) : r % RB;
        const uint8_t* bf0 = sm.slot(os) + kHalfBlocks * H * bfu;
        const float* z0 = sm.slot_z(os) + kHalfBlocks * H * M;
        float ai[TPW][NT][2];
#pragma unroll
        for (int tp = 0; tp < TPW; ++tp)
#pragma unroll
            for (int t = 0; t < NT; ++t) ai[tp][t][0] = ai[tp][t][1] = 0.0f;
        pn_block<TYPE, NT, TPW, kHalfBlocks * H + 0>(row0, tig, sel, bf0 + 0 * bfu, lane, live, rs, z0 + 0 * M, M,
                                                     ai);
        pn_block<TYPE, NT, TPW, kHalfBlocks * H + 1>(row0, tig, sel, bf0 + 1 * bfu, lane, live, rs, z0 + 1 * M, M,
                                                     ai);
        pn_block<TYPE, NT, TPW, kHalfBlocks * H + 2>(row0, tig, sel, bf0 + 2 * bfu, lane, live, rs, z0 + 2 * M, M,
                                                     ai);
        pn_block<TYPE, NT, TPW, kHalfBlocks * H + 3>(row0, tig, sel, bf0 + 3 * bfu, lane, live, rs, z0 + 3 * M, M,
                                                     ai);
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.empty(s));
        // the item's sums times 2^(24 - sigma) of its unit
        const float* so = sm.slot_so(os);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int m = 4 * t + tig;
            const float f = (m < M) ? so[m] : 0.0f;
#pragma unroll
            for (int tp = 0; tp < TPW; ++tp) {
                acc[tp][t][0] = fmaf(ai[tp][t][0], f, acc[tp][t][0]);
                acc[tp][t][1] = fmaf(ai[tp][t][1], f, acc[tp][t][1]);
            }
        }
    }
    if (ok && n_items > 0) emit();
    if (!ok && lane == 0) record_error(cx.err, kErrFullWait);
}

template <int TYPE, int NT, int TPW>
__global__ void __launch_bounds__(Cfg<TYPE, NT, TPW>::THREADS, 1) pn_gemv_kernel(const __grid_constant__ PnArgs a) {
    using C = Cfg<TYPE, NT, TPW>;
    constexpr int UK = C::UK;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    // builder jobs: one per row, or two (block halves) per row when there are fewer rows than builders
    const int parts = (a.M < C::NB) ? 2 : 1;
    const Smem sm{base,         smem_addr(base), a.NS,       a.RB,         a.M,           UK,
                  a.list_off,   a.part_off,      a.xs_off,   a.ring_off,   a.stage_off,   a.slot_bytes,
                  static_cast<uint32_t>(kUnitBlocks * C::bfu(a.M)), a.list_cap, a.M * parts};
    const Ctx cx{a.sc, a.X, a.Y, a.ws, a.cnt, a.err, a.N, a.K, a.M, a.NS, a.RB, a.flags};
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // this CTA's share of the items
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
        // ---------------- producer: one tensor-map copy per item ----------------
        if (lane == 0 && n_items > 0) {
            const uint64_t pol = l2_policy_evict_first();
            bool ok = true;
            int t_n = sc.tile_of(i0), u_n = sc.unit_of(i0);  // next item to request
            const int x_stage = (cx.flags & kXOverlap) ? a.x_stage : cx.NS;  // stages holding x at first
            auto issue = [&](int gi) {
                const int s = gi % cx.NS;
                if (gi >= cx.NS) {
                    if (!mbar_wait_bounded(sm.empty(s), ((gi / cx.NS) - 1) & 1)) return false;
                } else if (s >= x_stage) {
                    if (!mbar_wait_bounded(sm.x_free(), 0)) return false;
                }
                mbar_arrive_expect_tx(sm.full(s), static_cast<uint32_t>(kStageBytes));
                tma_load_2d(smem_addr(sm.stage(s)), &a.map, u_n * kUnitU32, t_n * kTileRows, sm.full(s), pol);
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
            int u_first = u_i, n_run = 0;  // the current share: first unit, items so far
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
                if (reduce_share<4 * NT>(cx, sm, buf, t_cur, u_first, n_run, lane)) {
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
        // (unit slot k = unit u0 + k mod U; jobs = (slot, row, block half)). Building only the
        // first unit here and the rest in the builder warps behind the consumers measured slower:
        // the prologue is mostly the x copy's latency, and two builder warps slow every item.
        if (n_items > 0) {
            const int u0 = sc.unit_of(i0);
            const int span = sc.span(i0, i1);
            const int pw = (warp < C::CW) ? warp : warp - C::BUILDER + C::CW;
            const int M = cx.M;
            const float* X = static_cast<const float*>(cx.X);
            float* xs = sm.xs(0);
            constexpr int CH = UK / 4;  // 16-byte chunks per row and unit
            auto copy = [&](int row) {     // x row slot row = k * M + m, by one warp
                const int k = row / M, m = row - k * M;
                int u = u0 + k;
                if (u >= sc.U) u -= sc.U;
                const float* src = X + static_cast<size_t>(m) * cx.K + static_cast<size_t>(u) * UK;
                const uint32_t dst = smem_addr(xs + static_cast<size_t>(row) * UK);
#pragma unroll
                for (int q = lane; q < CH; q += 32) cp_async16(dst + 16u * q, src + 4 * q);
            };
            const BuildLane<TYPE> bl(lane);
            const int rs = C::lg(M) * 16;
            const bool overlap = (a.flags & kXOverlap) != 0;
            auto job = [&](int i) {
                const int k = i / (2 * M), j = i - k * 2 * M;
                const int m = j >> 1, h = j & 1;
                build_row<TYPE, NT, 4>(sm.slot(k), sm.slot_z(k), sm.slot_so(k), xs + static_cast<size_t>(k * M + m) * UK,
                                       m, M, 4 * h, lane, bl, rs);
            };
            resident_prologue(pw, C::CW + C::NB, span * M, span * M * 2, overlap, copy, job);
            if (threadIdx.x == 0 && overlap) mbar_arrive(sm.x_free());
            if (warp < C::TG)
                consumer_loop<TYPE, NT, TPW, 0>(sm, cx, i0, n_items);
            else if (warp < C::CW)
                consumer_loop<TYPE, NT, TPW, 1>(sm, cx, i0, n_items);
        }
    } else if (warp >= C::BUILDER) {
        // ---------------- builders: operands of each run; jobs j = b, b + NB, .. ----------------
        // job j = row j / parts, block part j % parts; its x row is copied to x row slot j
        if (n_items > 0) {
            griddep_wait();  // X belongs to the previous grid until now
            const int b = warp - C::BUILDER;
            const float* X = static_cast<const float*>(cx.X);
            auto issue = [&](int u, int buf) {
                float* xb = sm.xs(buf);
                for (int j = b; j < sm.J; j += C::NB) {
                    const float* src = X + static_cast<size_t>(j / parts) * cx.K + static_cast<size_t>(u) * UK;
                    const uint32_t dst = smem_addr(xb + j * UK);
                    for (int q = lane; q < UK / 4; q += 32) cp_async16(dst + 16u * q, src + 4 * q);
                }
            };
            const BuildLane<TYPE> bl(lane);
            auto build = [&](int slot, int buf) {
                const float* xb = sm.xs(buf);
                for (int j = b; j < sm.J; j += C::NB) {
                    if (parts == 2)
                        build_row<TYPE, NT, 4>(sm.slot(slot), sm.slot_z(slot), sm.slot_so(slot), xb + j * UK, j >> 1,
                                               cx.M, 4 * (j & 1), lane, bl, C::lg(cx.M) * 16);
                    else
                        build_row<TYPE, NT, 8>(sm.slot(slot), sm.slot_z(slot), sm.slot_so(slot), xb + j * UK, j, cx.M,
                                               0, lane, bl, C::lg(cx.M) * 16);
                }
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
                consumer_loop<TYPE, NT, TPW, 0>(sm, cx, i0, n_items);
            else
                consumer_loop<TYPE, NT, TPW, 1>(sm, cx, i0, n_items);
        }
    }
    // the tiles this CTA completed: every warp sums some of them
    __syncthreads();
    finish_tiles(cx, sm, warp, C::THREADS / 32, lane);
}

// ---- host side --------------------------------------------------------------------------------------

constexpr int kDefaultStages = 3;

struct Plan {
    Sched sc{};
    bool publish = false;  // some tile is shared by several CTAs (the workspace is used)
    unsigned mode = 0;     // kResident, kXOverlap
    int NS = 0, RB = 0, XB = 0, x_stage = 0, list_cap = 0;
    uint32_t list_off = 0, part_off = 0, xs_off = 0, ring_off = 0, stage_off = 0, slot_bytes = 0, total = 0;
};

// Barriers, lists and row sums at the start; returns the first free (128-aligned) offset.
uint32_t head_layout(int bfu, int M, int NS, int RB, Plan& p) {
    p.list_cap = (p.sc.items + p.sc.G - 1) / p.sc.G;
    p.list_off = align_up(8u * (2u * NS + 2u * RB + 5u), 16);  // full, empty, op_full, op_empty, part x 4, x_free
    p.part_off = align_up(p.list_off + (2u * p.list_cap + 4u) * 4u, 16);
    p.slot_bytes = align_up(kUnitBlocks * static_cast<uint32_t>(bfu) + (kUnitBlocks + 1u) * M * 4u, 128);
    return align_up(p.part_off + 4u * M * kPartPitch * 4u, 128);
}

// Streaming layout: NS weight stages, RB operand slots and XB x buffers; false when it does not fit.
bool layout(int uk, int bfu, int M, int nb, int NS, int RB, int XB, Plan& p) {
    p.xs_off = head_layout(bfu, M, NS, RB, p);
    const uint32_t jobs = static_cast<uint32_t>(M) * (M < nb ? 2u : 1u);  // x rows per buffer
    p.ring_off = align_up(p.xs_off + static_cast<uint32_t>(XB) * jobs * uk * 4u, 128);
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
bool layout_resident(int uk, int bfu, int M, int NS, bool overlap, Plan& p) {
    int span = 0;
    for (int c = 0; c < p.sc.G; ++c) span = std::max(span, p.sc.span(p.sc.first(c), p.sc.first(c + 1)));
    uint64_t off = head_layout(bfu, M, NS, 0, p);
    const uint64_t xbytes = static_cast<uint64_t>(span) * M * uk * 4u;
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

// Resident operands with the deepest weight ring up to ns_max (at least 3 stages), x in its own
// region when that fits (measured faster than a deeper ring whose last stages wait for x), else
// in the weight stages.
bool fit_resident(int uk, int bfu, int M, int ns_req, Plan& p) {
    const int ns_max = ns_req > 0 ? ns_req : kDefaultStages, ns_lo = ns_req > 0 ? ns_req : 3;
    for (bool overlap : {false, true})
        for (int ns = ns_max; ns >= ns_lo; --ns)
            if (layout_resident(uk, bfu, M, ns, overlap, p)) return true;
    return false;
}

// Streaming ring: the deepest weight ring up to ns_max (at least 3 stages when possible), then
// the deepest x prefetch and operand ring that fit; rb_req > 0 forces the ring's slots.
bool fit_stream(int uk, int bfu, int M, int nb, int ns_req, int rb_req, Plan& p) {
    const int ns_max = ns_req > 0 ? ns_req : kDefaultStages;
    for (int ns_min : {3, 2})
        for (int xb : {4, 2, 1})
            for (int rb : {3, 2}) {
                if (rb_req > 0 && rb != 3) continue;
                const int r = rb_req > 0 ? std::min(std::max(rb_req, 2), 4) : rb;  // one slot would deadlock
                for (int ns = ns_max; ns >= (ns_req > 0 ? ns_req : ns_min); --ns)
                    if (layout(uk, bfu, M, nb, ns, r, xb, p)) return true;
            }
    return false;
}

// Grid, item order and layout. Tile-major items with resident operands when they fit: grid of
// one CTA per SM (stream-K) or, with fewer row tiles than SMs, one CTA per tile (nothing to
// reduce across CTAs), whichever has the smaller estimate of (items of the busiest CTA) +
// (cross-CTA reduction tail). Otherwise (wide batches) one CTA per SM with grouped unit-major
// items (the smallest group whose operands fit, resident) or, when that does not fit or
// order = 1, tile-major items with the streaming ring. rb_req > 0 forces the streaming ring,
// order = 2 the grouped order.
bool make_plan(int uk, int bfu, int M, int nb, int64_t T, int64_t U, int sms, bool grid_forced, int ns_req,
               int rb_req, int order, Plan& p) {
    const int64_t items = T * U;
    const int64_t G0 = std::min<int64_t>(sms, items);
    int64_t cands[2] = {G0, 0};
    if (!grid_forced && T < sms) cands[1] = T;
    auto base = [&](int64_t G) {
        Plan q;
        q.sc.items = static_cast<int>(items);
        q.sc.T = static_cast<int>(T);
        q.sc.U = static_cast<int>(U);
        q.sc.G = static_cast<int>(G);
        q.sc.tile_major = 1;
        q.sc.tg = 1;
        return q;
    };
    auto publishes = [](const Plan& q) {
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
            Plan q = base(G);
            if (!fit_resident(uk, bfu, M, ns_req, q)) continue;
            q.publish = publishes(q);
            const double cost = static_cast<double>((items + G - 1) / G) + (q.publish ? 2.5 : 0.0);
            if (!found || cost < best) {
                best = cost;
                p = q;
                found = true;
            }
        }
    if (found) return true;
    if (rb_req <= 0 && order != 1 && T > 1 && U > 1) {
        for (int64_t tg : {2, 4, 8, 16, 32, 64, 128}) {
            Plan q = base(G0);
            q.sc.tile_major = 0;
            q.sc.tg = static_cast<int>(std::min<int64_t>(tg, T));
            if (fit_resident(uk, bfu, M, ns_req, q)) {
                q.publish = publishes(q);
                p = q;
                return true;
            }
            if (tg >= T) break;
        }
    }
    Plan q = base(G0);
    if (!fit_stream(uk, bfu, M, nb, ns_req, rb_req, q)) return false;
    q.publish = publishes(q);
    p = q;
    return true;
}

// Environment override PNQ_PN_CFG="tpw,grid,rb,ns,order,pf" (fields 0 = automatic), read once.
MmaConfig env_config() {
    static MmaConfig cfg = [] {
        MmaConfig c{0, 0, 0, 0, 0, 0};
        if (const char* s = std::getenv("PNQ_PN_CFG")) {
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

template <int TYPE, int NT, int TPW>
cudaError_t launch_cfg(PnArgs& a, const MmaConfig& cfg, bool static_weights, cudaStream_t stream,
                       const ExtWorkspace& ext) {
    using C = Cfg<TYPE, NT, TPW>;
    Plan p;
    const int cap = cfg.grid > 0 ? std::min(cfg.grid, device_sm_count()) : device_sm_count();
    if (!make_plan(C::UK, C::bfu(a.M), a.M, C::NB, a.sc.T, a.sc.U, cap, cfg.grid > 0, cfg.ns, cfg.rb, cfg.order, p))
        return cudaErrorNotSupported;
    auto kern = pn_gemv_kernel<TYPE, NT, TPW>;
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
        // the caller's scratch: too small only matters when CTAs share tiles
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
    // may begin while the previous grid in the stream finishes (see griddep_wait in the kernel)
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, kern, a);
}

template <int TYPE>
cudaError_t launch_typed(PnArgs& a, const MmaConfig& cfg, bool static_weights, cudaStream_t stream,
                         const ExtWorkspace& ext) {
    const int nt = (2 * a.M + 7) / 8;
    // one tile per warp (16 consumer warps) for the matrix-vector range; two tiles per warp
    // (8 consumer warps, B fragments reused across the tiles) for wider batches
    const int tpw = cfg.tpw > 0 ? cfg.tpw : (nt == 1 ? 1 : 2);
    if (nt == 1) return tpw == 1 ? launch_cfg<TYPE, 1, 1>(a, cfg, static_weights, stream, ext)
                                 : launch_cfg<TYPE, 1, 2>(a, cfg, static_weights, stream, ext);
    if (nt == 2) return tpw == 1 ? launch_cfg<TYPE, 2, 1>(a, cfg, static_weights, stream, ext)
                                 : launch_cfg<TYPE, 2, 2>(a, cfg, static_weights, stream, ext);
    return tpw == 1 ? launch_cfg<TYPE, 4, 1>(a, cfg, static_weights, stream, ext)
                    : launch_cfg<TYPE, 4, 2>(a, cfg, static_weights, stream, ext);
}

}  // namespace

cudaError_t launch_pn_gemv_mma(int type, const uint8_t* W, int64_t N, int64_t K, const float* X, int M, float* Y,
                               int* err, MmaConfig cfg, bool static_weights, cudaStream_t stream,
                               const ExtWorkspace& ext) {
    if (N == 0) return cudaSuccess;
    const int blk = (type == kTypePn3t) ? 80 : 64;
    const int64_t nb = K / blk;
    if (nb % kUnitBlocks != 0 || M < 1 || M > 16) return cudaErrorNotSupported;
    const int64_t U = nb / kUnitBlocks, T = (N + kTileRows - 1) / kTileRows;
    if (N > INT32_MAX || K > INT32_MAX || U * kUnitU32 > INT32_MAX || T * kTileRows > INT32_MAX ||
        T * U > INT32_MAX)
        return cudaErrorNotSupported;
    if (reinterpret_cast<uintptr_t>(W) % 16 != 0 || reinterpret_cast<uintptr_t>(X) % 16 != 0)
        return cudaErrorNotSupported;
    PnArgs a{};
    if (!encode_u32_map(&a.map, W, N, nb * kBlockBytes / 4, kUnitU32, kTileRows)) return cudaErrorNotSupported;
    a.X = X;
    a.Y = Y;
    a.err = err;
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.M = M;
    a.sc.T = static_cast<int>(T);
    a.sc.U = static_cast<int>(U);
    a.sc.items = static_cast<int>(T * U);
    const MmaConfig c =
        (cfg.tpw > 0 || cfg.grid > 0 || cfg.rb > 0 || cfg.ns > 0 || cfg.order > 0 || cfg.pf > 0) ? cfg : env_config();
    return (type == kTypePn3t) ? launch_typed<kTypePn3t>(a, c, static_weights, stream, ext)
                               : launch_typed<kTypePn4t>(a, c, static_weights, stream, ext);
}

}  // namespace pnq
