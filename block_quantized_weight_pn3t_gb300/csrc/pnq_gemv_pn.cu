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
// Items and schedule (stream-K). The weight matrix is cut into items of 128 rows x one K unit
// of 8 blocks (272 bytes per row). Items are numbered unit-major (item = u * T + t for row tile
// t of T) and every CTA of a persistent grid (one per SM) takes an equal contiguous share, so
// all SMs stream the same number of bytes and a CTA's items touch at most a few K units.
//
// Memory pipeline. One producer thread loads one item per stage with a 2-D tensor-map copy
// (box 272 bytes x 128 rows, L2 evict-first; rows past N read as zeros) into an NS-stage ring
// under mbarriers; at start it also copies the CTA's slice of x (fp32) into the last stages.
// With the static-weights flag the first stages are requested before the previous grid in the
// stream has finished.
//
// Decode and multiply (consumer warps). Warp = TPW tiles of 16 rows x half a unit (4 blocks).
// A 32-bit word of a block holds two codes at the same shift in its two 16-bit halves; masking
// out one such pair leaves in each half the exact fp16 subnormal n * 2^-24 * 8^j (pn3t; 16^j
// for pn4t, j = position of the pair): one AND per two weights gives an mma A register. Lane
// (g, c) of the warp uses words c and c + 4 of rows g and g + 8; the k order inside a block is
// free as long as B uses the same order, so the 2-byte aligned words of even blocks are read as
// aligned words pairing the high half of word i-1 with the low half of word i (one PRMT).
//
// B operand: x times 8^-j (16^-j) times 2^sigma (per CTA and activation row, so that max|x| *
// 2^sigma lies in [2^14, 2^15)), split into fp16 hi + lo parts (~22 bits) that take mma
// columns 2m and 2m + 1 (NT = ceil(2M / 8) n8 tiles). The fragments of the CTA's blocks are
// built once in shared memory in register order.
//
// Block scale and zero point: acc += d * (c - Z) per block, Z = z * (sum over the block of B
// times 2^-24 * 8^j), precomputed beside B in fp32.
//
// Reduction. At the end of an item the consumer warps leave their row sums (two halves) in
// shared memory; a reducer warp adds them, writes the item's rows to a workspace slot and
// counts the item on its row tile; the CTA that brings a tile's count to U sums the tile's U
// slots in unit order (so the result does not depend on timing) and writes Y.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
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
    static constexpr int TG = 8 / TPW;             // tile groups per half
    static constexpr int CW = 2 * TG;              // consumer warps
    static constexpr int PRODUCER = CW, REDUCER = CW + 1;
    static constexpr int THREADS = 32 * (CW + 2);
    static constexpr int NCT = 32 * CW;            // consumer threads
    static constexpr int BFU = NT * 256 * STEPS;   // fragment bytes per block
};

struct PnArgs {
    CUtensorMap map;  // weights as u32 [N][row_bytes / 4], box {68, 128}
    const float* X;
    float* Y;
    float* ws;       // partial rows [T][U][M][128]: slot (t, u) = the share of tile t starting at unit u
    uint32_t* cnt;   // [T] shares counted per row tile (zero between launches)
    int* err;
    Sched sc;
    int N, K, M, NS, x_stage, xpitch;
    unsigned flags;
    uint32_t bar_off, misc_off, z_off, part_off, b_off, stage_off, list_off;
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

// Shared-memory regions (offsets from the 1024-aligned base).
struct Smem {
    uint8_t* base;
    uint32_t bar0;  // shared address of barrier 0
    int NS;
    uint32_t misc_off, z_off, part_off, b_off, stage_off, list_off;
    __device__ uint32_t full(int s) const { return bar0 + 8u * s; }
    __device__ uint32_t empty(int s) const { return bar0 + 8u * (NS + s); }
    __device__ uint32_t x_free() const { return bar0 + 8u * (2 * NS + 1); }
    __device__ uint32_t part_full(int b) const { return bar0 + 8u * (2 * NS + 2 + b); }
    __device__ uint32_t part_free(int b) const { return bar0 + 8u * (2 * NS + 4 + b); }
    __device__ uint32_t* maxbits() const { return reinterpret_cast<uint32_t*>(base + misc_off); }
    __device__ float* sig_in() const { return reinterpret_cast<float*>(base + misc_off + 64); }
    __device__ float* sig_out() const { return reinterpret_cast<float*>(base + misc_off + 128); }
    __device__ float* z() const { return reinterpret_cast<float*>(base + z_off); }
    __device__ float* part() const { return reinterpret_cast<float*>(base + part_off); }
    __device__ uint8_t* b() const { return base + b_off; }
    __device__ uint8_t* stage(int s) const { return base + stage_off + static_cast<uint32_t>(s) * kStageBytes; }
    // tiles whose partial shares wait to be counted, tiles this CTA completes (list_cap entries
    // each, list_cap >= the items of any CTA), and the number of the latter
    int list_cap;
    __device__ int* n_finish() const { return reinterpret_cast<int*>(base + list_off); }
    __device__ int* pending() const { return reinterpret_cast<int*>(base + list_off) + 4; }
    __device__ int* finish() const { return reinterpret_cast<int*>(base + list_off) + 4 + list_cap; }
};

// A register (two halves) holding code 1 at slice j's position: the fp16 subnormal
// 2^-24 * 8^j (pn3t) or 2^-24 * 16^j (pn4t) in both halves.
template <int TYPE>
__device__ __forceinline__ uint32_t code_one(int j) {
    const int jj = (TYPE == kTypePn3t) ? (j < 3 ? j : j - 3) : (j & 1);
    return 0x00010001u << (PnFmt<TYPE>::BITS * jj);
}

// B fragments of one block for every n8 tile: lanes whose column is in use load their records,
// the others hold zeros.
template <int TYPE, int NT>
__device__ __forceinline__ void load_bfrag(const uint8_t* bf, int lane, const bool (&live)[NT],
                                           uint32_t (&b)[NT][PnFmt<TYPE>::PAIRS][2]) {
    constexpr int STEPS = PnFmt<TYPE>::PAIRS;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const uint8_t* base = bf + t * 256 * STEPS;
#pragma unroll
        for (int q = 0; q < STEPS / 2; ++q) {
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (live[t]) v = *reinterpret_cast<const uint4*>(base + q * 512 + lane * 16);
            b[t][2 * q][0] = v.x;
            b[t][2 * q][1] = v.y;
            b[t][2 * q + 1][0] = v.z;
            b[t][2 * q + 1][1] = v.w;
        }
        if constexpr (STEPS & 1) {
            uint2 v = make_uint2(0u, 0u);
            if (live[t]) v = *reinterpret_cast<const uint2*>(base + (STEPS / 2) * 512 + lane * 8);
            b[t][STEPS - 1][0] = v.x;
            b[t][STEPS - 1][1] = v.y;
        }
    }
}

// sigma per activation row, the B fragments and the per-block zero-point sums for the CTA's
// nblk blocks (consumer threads only).
template <int TYPE, int NT, int TPW>
__device__ __forceinline__ void fill_operands(const Smem& sm, const float* X, int K, int U, int u0, int span,
                                              float* xs, int xpitch, int M) {
    using F = PnFmt<TYPE>;
    using C = Cfg<TYPE, NT, TPW>;
    constexpr int STEPS = F::PAIRS;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nblk = span * kUnitBlocks;
    uint32_t* maxbits = sm.maxbits();
    float* sig_in = sm.sig_in();
    float* sig_out = sm.sig_out();
    // x: the CTA's K units (slots 0..span-1 = units u0, u0+1, .. mod U) of every row, straight
    // from global memory (L2 only: X may have been written by the previous grid), into shared
    // memory at pitch xpitch; max |x| per row on the way (a non-negative float's bits order like
    // its value)
    constexpr int UK = kUnitBlocks * F::BLK;
    const int vec = span * (UK / 4);
    for (int m = 0; m < M; ++m) {
        const float* xg = X + static_cast<size_t>(m) * K;
        float* xd = xs + m * xpitch;
        uint32_t mx = 0;
        for (int q = tid; q < vec; q += C::NCT) {
            const int sl = q / (UK / 4);
            int u = u0 + sl;
            if (u >= U) u -= U;
            const int off = 4 * q - sl * UK;
            const float4 v = __ldcg(reinterpret_cast<const float4*>(xg + static_cast<size_t>(u) * UK + off));
            *reinterpret_cast<float4*>(xd + sl * UK + off) = v;
            mx = max(mx, max(max(__float_as_uint(v.x) & 0x7FFFFFFFu, __float_as_uint(v.y) & 0x7FFFFFFFu),
                             max(__float_as_uint(v.z) & 0x7FFFFFFFu, __float_as_uint(v.w) & 0x7FFFFFFFu)));
        }
        mx = __reduce_max_sync(0xffffffffu, mx);
        if (lane == 0) atomicMax(&maxbits[m], mx);
    }
    fence_proxy_async_smem();  // these bytes are later overwritten by tensor-map copies
    named_sync(1, C::NCT);
    if (tid < M) {
        const uint32_t bits = maxbits[tid];
        const int E = static_cast<int>(bits >> 23);
        int sg = (bits == 0 || E >= 255) ? 0 : 141 - E;  // max < 2^(E-126)
        sg = min(100, max(-100, sg));
        sig_in[tid] = exp2i(sg);
        sig_out[tid] = exp2i(24 - sg);  // undoes sigma and the 2^-24 of the subnormal codes
    }
    named_sync(1, C::NCT);
    // B fragments: one item per (block, pair of slices, lane column c), rows m inside. For slices
    // 2p and 2p + 1 the item builds the registers b0 (decode register c) and b1 (register c + 4)
    // of row m's hi column 2m and lo column 2m + 1 and stores them as the two 16-byte lane
    // records (lane = 4 * (column % 8) + c; an odd last slice has 8-byte records).
    uint8_t* bbase = sm.b();
    constexpr int PAIRS = (STEPS + 1) / 2;
    const int items = nblk * PAIRS * 4;
    for (int it = tid; it < items; it += C::NCT) {
        const int c = it & 3, rest = it >> 2;
        const int pr = rest % PAIRS, blk = rest / PAIRS;
        const int odd = blk & 1;
        const bool single = (STEPS & 1) && pr == PAIRS - 1;  // the odd last slice alone
        for (int m = 0; m < M; ++m) {
            const float* xb = xs + m * xpitch + blk * F::BLK;
            uint32_t hi[4] = {0u, 0u, 0u, 0u}, lo[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int q = 0; q < 4; ++q) {  // q = 2 * (slice - 2pr) + register
                const int st = 2 * pr + (q >> 1), i = c + 4 * (q & 1);
                if (st < STEPS) {
                    const float sc = sig_in[m] * step_scale<TYPE>(st);
                    const float v0 = xb[pn_elem(F::CPW, odd, i, st, 0)] * sc;
                    const float v1 = xb[pn_elem(F::CPW, odd, i, st, 1)] * sc;
                    const __half h0 = __float2half_rn(v0), h1 = __float2half_rn(v1);
                    hi[q] = pack_half2(h0, h1);
                    lo[q] = pack_half2(__float2half_rn(v0 - __half2float(h0)), __float2half_rn(v1 - __half2float(h1)));
                }
            }
            const int n = 2 * m;  // hi column; the lo column n + 1 is in the same n8 tile
            uint8_t* tb = bbase + blk * C::BFU + (n >> 3) * 256 * STEPS + pr * 512;
            const int lh = ((n & 7) << 2) | c, ll = (((n + 1) & 7) << 2) | c;
            if (single) {
                *reinterpret_cast<uint2*>(tb + lh * 8) = make_uint2(hi[0], hi[1]);
                *reinterpret_cast<uint2*>(tb + ll * 8) = make_uint2(lo[0], lo[1]);
            } else {
                *reinterpret_cast<uint4*>(tb + lh * 16) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(tb + ll * 16) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
        }
    }
    named_sync(1, C::NCT);
    // Z = z * sum over the block of (2^-24 * 8^j) * B, on the tensor core: an A operand with code
    // 1 at slice j's position in every row and k (the subnormal 2^-24 * 8^j) sums B the same way
    // the main loop's mma sums n * 2^-24 * 8^j * B. One warp per block.
    float* z = sm.z();
    const int g = lane >> 2, tig = lane & 3;
    bool live[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) live[t] = (8 * t + g) < 2 * M;
    for (int blk = warp; blk < nblk; blk += C::CW) {
        uint32_t b[NT][STEPS][2];
        load_bfrag<TYPE, NT>(bbase + blk * C::BFU, lane, live, b);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            float c[4];
#pragma unroll
            for (int j = 0; j < STEPS; ++j) {
                const uint32_t one = code_one<TYPE>(j);
                if (j == 0)
                    mma_f16_16816_z(c, one, one, one, one, b[t][j][0], b[t][j][1]);
                else
                    mma_f16_16816(c, one, one, one, one, b[t][j][0], b[t][j][1]);
            }
            const int m = 4 * t + tig;
            if (g == 0 && m < M) z[blk * M + m] = static_cast<float>(F::Z) * (c[0] + c[1]);
        }
    }
    named_sync(1, C::NCT);
}

// One block B (of the unit, compile time) for the warp's TPW tiles: decode, multiply, fold
// d * (c - Z) into acc[tile][t][row half].
template <int TYPE, int NT, int TPW, int B>
__device__ __forceinline__ void pn_block(const uint8_t* const (&row0)[TPW], int tig, uint32_t sel,
                                         const uint8_t* bf, int lane, const bool (&live)[NT], const float* zb, int M,
                                         float (&acc)[TPW][NT][2]) {
    using F = PnFmt<TYPE>;
    constexpr int STEPS = F::PAIRS;
    constexpr int OFF = kBlockBytes * B;
    constexpr int SH = (TYPE == kTypePn3t) ? 9 : 8;
    // B fragments (columns past 2M are zero and are not read)
    uint32_t b[NT][STEPS][2];
    load_bfrag<TYPE, NT>(bf, lane, live, b);
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
__device__ __forceinline__ void consumer_loop(const Smem& sm, const Ctx& cx, int i0, int n_items, int u0) {
    using C = Cfg<TYPE, NT, TPW>;
    const Sched& sc = cx.sc;
    const int M = cx.M, NS = cx.NS, U = sc.U;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tig = lane & 3;
    const int tg = warp % C::TG;  // tile group: rows 16 * TPW * tg ..
    const uint32_t sel = (tig == 0) ? 0x5432u : 0x3210u;  // even blocks: register 0 pairs words 0 and 7
    bool live[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) live[t] = (8 * t + g) < 2 * M;
    const float* z = sm.z();
    const float* sig_out = sm.sig_out();
    float* part = sm.part();
    bool ok = true;
    float acc[TPW][NT][2];
#pragma unroll
    for (int tp = 0; tp < TPW; ++tp)
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[tp][t][0] = acc[tp][t][1] = 0.0f;
    int e = 0;  // row sums handed to the reducer so far
    // hand the row sums of the tile just finished to the reducer (scaled back), then clear them
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
                    dst[0] = acc[tp][t][0] * sig_out[m];
                    dst[8] = acc[tp][t][1] * sig_out[m];
                }
                acc[tp][t][0] = acc[tp][t][1] = 0.0f;
            }
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.part_full(buf));
        ++e;
    };
    int t_i = sc.tile_of(i0), u_i = sc.unit_of(i0);
    int cur_t = t_i;
    for (int gi = 0; gi < n_items && ok; ++gi, next_item(sc, t_i, u_i)) {
        if (t_i != cur_t) {
            emit();
            if (!ok) break;
            cur_t = t_i;
        }
        const int slot = (u_i >= u0) ? u_i - u0 : u_i - u0 + U;
        const int s = gi % NS;
        if (!mbar_wait_warp(sm.full(s), (gi / NS) & 1)) {
            ok = false;
            break;
        }
        const uint8_t* stage = sm.stage(s);
        const uint8_t* row0[TPW];
#pragma unroll
        for (int tp = 0; tp < TPW; ++tp) row0[tp] = stage + (16 * (TPW * tg + tp) + g) * kUnitBytes;
        const int blk0 = slot * kUnitBlocks + kHalfBlocks * H;
        const uint8_t* bf0 = sm.b() + blk0 * C::BFU;
        const float* z0 = z + blk0 * M;
        pn_block<TYPE, NT, TPW, kHalfBlocks * H + 0>(row0, tig, sel, bf0 + 0 * C::BFU, lane, live, z0 + 0 * M, M, acc);
        pn_block<TYPE, NT, TPW, kHalfBlocks * H + 1>(row0, tig, sel, bf0 + 1 * C::BFU, lane, live, z0 + 1 * M, M, acc);
        pn_block<TYPE, NT, TPW, kHalfBlocks * H + 2>(row0, tig, sel, bf0 + 2 * C::BFU, lane, live, z0 + 2 * M, M, acc);
        pn_block<TYPE, NT, TPW, kHalfBlocks * H + 3>(row0, tig, sel, bf0 + 3 * C::BFU, lane, live, z0 + 3 * M, M, acc);
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.empty(s));
    }
    if (ok && n_items > 0) emit();
    if (!ok && lane == 0) record_error(cx.err, kErrFullWait);
}

template <int TYPE, int NT, int TPW>
__global__ void __launch_bounds__(Cfg<TYPE, NT, TPW>::THREADS, 1) pn_gemv_kernel(const __grid_constant__ PnArgs a) {
    using F = PnFmt<TYPE>;
    using C = Cfg<TYPE, NT, TPW>;
    constexpr int UK = kUnitBlocks * F::BLK;  // weights of a row per unit
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const Smem sm{base,        smem_addr(base + a.bar_off), a.NS,       a.misc_off, a.z_off, a.part_off,
                  a.b_off,     a.stage_off,                 a.list_off, a.list_cap};
    const Ctx cx{a.sc, a.X, a.Y, a.ws, a.cnt, a.err, a.N, a.K, a.M, a.NS, a.x_stage, a.xpitch, a.flags};
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // this CTA's share of the items, and the K units it touches (slot = (u - u0) mod U)
    const Sched& sc = cx.sc;
    const int i0 = sc.first(blockIdx.x), i1 = sc.first(blockIdx.x + 1);
    const int n_items = static_cast<int>(i1 - i0);
    const int u0 = n_items > 0 ? sc.unit_of(i0) : 0;
    const int span = sc.span(i0, i1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.NS; ++s) {
            mbar_init(sm.full(s), 1);
            mbar_init(sm.empty(s), C::CW);
        }
        mbar_init(sm.x_free(), 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(sm.part_full(b), C::CW);
            mbar_init(sm.part_free(b), 1);
        }
        mbar_fence_init();
        griddep_launch_dependents();
    }
    if (threadIdx.x < 16) sm.maxbits()[threadIdx.x] = 0u;
    if (threadIdx.x == 0) *sm.n_finish() = 0;
    __syncthreads();

    if (warp == C::PRODUCER) {
        // ---------------- producer: x slice + one tensor-map copy per item ----------------
        if (lane == 0 && n_items > 0) {
            const uint64_t pol = l2_policy_evict_first();
            bool ok = true;
            int t_n = sc.tile_of(i0), u_n = sc.unit_of(i0);  // next item to request
            auto issue = [&](int gi) {
                const int s = gi % cx.NS;
                if (gi >= cx.NS) {
                    if (!mbar_wait_bounded(sm.empty(s), ((gi / cx.NS) - 1) & 1)) return false;
                } else if (s >= cx.x_stage) {
                    if (!mbar_wait_bounded(sm.x_free(), 0)) return false;
                }
                mbar_arrive_expect_tx(sm.full(s), static_cast<uint32_t>(kStageBytes));
                tma_load_2d(smem_addr(sm.stage(s)), &a.map, u_n * kUnitU32, t_n * kTileRows, sm.full(s), pol);
                next_item(sc, t_n, u_n);
                return true;
            };
            int gi = 0;
            if (cx.flags & kStaticWeights) {
                // the weights are not written by earlier work in the stream: start streaming
                // them into the stages that will not hold x before the previous grid completes
                for (; ok && gi < min(n_items, cx.x_stage); ++gi) ok = issue(gi);
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
    } else {
        // ---------------- consumer warps ----------------
        if (n_items > 0) {
            griddep_wait();  // X belongs to the previous grid until now
            float* xs = reinterpret_cast<float*>(sm.stage(cx.x_stage));
            fill_operands<TYPE, NT, TPW>(sm, static_cast<const float*>(cx.X), cx.K, sc.U, u0, span, xs, cx.xpitch, cx.M);
            if (threadIdx.x == 0) mbar_arrive(sm.x_free());  // the x stages may now take weights
            if (warp < C::TG)
                consumer_loop<TYPE, NT, TPW, 0>(sm, cx, i0, n_items, u0);
            else
                consumer_loop<TYPE, NT, TPW, 1>(sm, cx, i0, n_items, u0);
        }
    }
    // the tiles this CTA completed: every warp sums some of them
    __syncthreads();
    const int nf = *sm.n_finish();
    for (int k = warp; k < nf; k += C::THREADS / 32) finish_tile(cx, sm.finish()[k], lane);
}

// ---- host side --------------------------------------------------------------------------------------

struct Plan {
    Sched sc{};
    bool publish = false;  // some tile is shared by several CTAs (the workspace is used)
    int NS = 0, x_stage = 0, span_max = 0, xpitch = 0, list_cap = 0;
    uint32_t bar_off = 0, misc_off = 0, list_off = 0, z_off = 0, part_off = 0, b_off = 0, stage_off = 0, total = 0;
};

// Shared-memory layout and stage count for one item order; false when it does not fit.
bool layout(int blk_weights, int bfu, int M, int ns_req, Plan& p) {
    p.span_max = 0;
    for (int c = 0; c < p.sc.G; ++c) p.span_max = std::max(p.span_max, p.sc.span(p.sc.first(c), p.sc.first(c + 1)));
    const uint32_t nblk = static_cast<uint32_t>(p.span_max) * kUnitBlocks;
    p.xpitch = static_cast<int>(nblk) * blk_weights + 4;
    p.bar_off = 0;
    p.misc_off = 8u * (2 * kMaxStages + 6);
    p.list_cap = (p.sc.items + p.sc.G - 1) / p.sc.G;
    p.list_off = align_up(p.misc_off + 192u, 16);
    p.z_off = align_up(p.list_off + (2u * p.list_cap + 4u) * 4u, 16);
    p.part_off = align_up(p.z_off + nblk * M * 4u, 16);
    p.b_off = align_up(p.part_off + 4u * M * kPartPitch * 4u, 128);
    p.stage_off = align_up(p.b_off + nblk * static_cast<uint32_t>(bfu), 1024);
    const uint64_t xbytes = static_cast<uint64_t>(M) * p.xpitch * 4u;
    const int x_stages = static_cast<int>((xbytes + kStageBytes - 1) / kStageBytes);
    for (int ns = kMaxStages; ns >= 2; --ns) {
        if (ns_req > 0 && ns != ns_req) continue;
        const uint64_t total = p.stage_off + static_cast<uint64_t>(ns) * kStageBytes;
        // at least three stages unless forced, and one stage free of x when the ring allows it
        if (total + 1024u <= kSmemLimit && ns >= x_stages && (ns_req > 0 || ns >= 3)) {
            p.NS = ns;
            p.x_stage = ns - x_stages;
            p.total = static_cast<uint32_t>(total);
            return true;
        }
    }
    return false;
}

// Grid, item order, stage count and layout. Candidates: one CTA per SM (stream-K), and one CTA
// per row tile when there are fewer tiles than SMs (every tile whole, nothing to reduce across
// CTAs). Tile-major when the operands of a share fit, else unit-major. Picks the smallest
// estimate of (items of the busiest CTA) x (time per item) + (cross-CTA reduction tail).
bool make_plan(int blk_weights, int bfu, int M, int64_t T, int64_t U, int sms, bool grid_forced, int ns_req, Plan& p) {
    const int64_t items = T * U;
    int64_t cands[2] = {std::min<int64_t>(sms, items), 0};
    if (!grid_forced && T < sms) cands[1] = T;
    bool found = false;
    double best = 0.0;
    for (int64_t G : cands) {
        if (G <= 0) continue;
        for (int tm = 1; tm >= 0; --tm) {
            Plan q;
            q.sc.items = items;
            q.sc.T = static_cast<int>(T);
            q.sc.U = static_cast<int>(U);
            q.sc.G = static_cast<int>(G);
            q.sc.tile_major = tm;
            if (!layout(blk_weights, bfu, M, ns_req, q)) continue;
            bool publish = false;
            for (int c = 1; c < G && !publish; ++c) publish = q.sc.tile_of(q.sc.first(c)) == q.sc.tile_of(q.sc.first(c) - 1);
            if (!tm && U > 1) publish = true;
            const double cost = static_cast<double>((items + G - 1) / G) + (publish ? 2.5 : 0.0);
            if (!found || cost < best) {
                best = cost;
                q.publish = publish;
                p = q;
                found = true;
            }
            break;  // unit-major only when tile-major does not fit
        }
    }
    return found;
}

// Environment override PNQ_PN_CFG="tpw,grid,_,ns" (fields 0 = automatic), read once.
MmaConfig env_config() {
    static MmaConfig cfg = [] {
        MmaConfig c{0, 0, 0, 0};
        if (const char* s = std::getenv("PNQ_PN_CFG")) {
            int v[4] = {0, 0, 0, 0};
            int n = 0;
            const char* p = s;
            while (*p && n < 4) {
                v[n++] = static_cast<int>(std::strtol(p, const_cast<char**>(&p), 10));
                if (*p == ',') ++p;
            }
            c = MmaConfig{v[0], v[1], v[2], v[3]};
        }
        return c;
    }();
    return cfg;
}

template <int TYPE, int NT, int TPW>
cudaError_t launch_cfg(PnArgs& a, const MmaConfig& cfg, bool static_weights, cudaStream_t stream,
                       const ExtWorkspace& ext) {
    using F = PnFmt<TYPE>;
    using C = Cfg<TYPE, NT, TPW>;
    Plan p;
    const int cap = cfg.S > 0 ? std::min(cfg.S, device_sm_count()) : device_sm_count();
    if (!make_plan(F::BLK, C::BFU, a.M, a.sc.T, a.sc.U, cap, cfg.S > 0, cfg.ns, p)) return cudaErrorNotSupported;
    auto kern = pn_gemv_kernel<TYPE, NT, TPW>;
    static bool opted[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!opted[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemLimit));
        if (e != cudaSuccess) return e;
        opted[dev] = true;
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
    a.x_stage = p.x_stage;
    a.xpitch = p.xpitch;
    a.flags = static_weights ? kStaticWeights : 0u;
    a.bar_off = p.bar_off;
    a.misc_off = p.misc_off;
    a.list_off = p.list_off;
    a.list_cap = p.list_cap;
    a.z_off = p.z_off;
    a.part_off = p.part_off;
    a.b_off = p.b_off;
    a.stage_off = p.stage_off;
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
    const int tpw = cfg.rw > 0 ? cfg.rw : (nt == 1 ? 1 : 2);
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
    const MmaConfig c = (cfg.rw > 0 || cfg.S > 0 || cfg.ns > 0) ? cfg : env_config();
    return (type == kTypePn3t) ? launch_typed<kTypePn3t>(a, c, static_weights, stream, ext)
                               : launch_typed<kTypePn4t>(a, c, static_weights, stream, ext);
}

}  // namespace pnq
