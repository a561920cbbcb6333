// pnq_gemv_pn.cu -- tensor-core GEMV straight from pn3t / pn4t 34-byte blocks (fast path).
//
// Computes Y[m][n] = sum_k w[n][k] x[m][k], 1 <= M <= 16, with w decoded in registers just
// before the multiply ("PN weight format", sections Block layout and Value).
//
// Work split. Persistent grid, one wave: clusters of S CTAs (S = 1, 2, 4 or 8), one CTA per
// SM. Weight rows are cut into 16-row tiles; each cluster owns a balanced contiguous range of
// tiles and streams it in passes of 4 tiles (64 rows); CTA rank q owns the q-th slice of K.
//
// Memory pipeline. One producer thread issues 2-D tensor-map copies: a stage is 16 blocks of
// 64 rows, loaded as two 64 x 272-byte boxes (272 bytes = 8 blocks, a multiple of 16 and an odd
// number of 16-byte lines, so a warp's 8 row groups hit distinct banks). Ragged last passes
// use 16-row boxes. NS stages ring under mbarriers, L2 evict-first. At start the producer
// also copies the CTA's slice of x (fp32) into the last stages of the ring.
//
// Compute. RW consumer warps (8 for M <= 4, else 4) split every stage along K: each takes its
// own 16/RW blocks for all four tiles, so each block's B fragments feed four independent mma
// chains. The decode is one AND per pair of weights: a 32-bit word holds two codes at the same shift in
// its two 16-bit halves, and with a zero fp16 exponent field the masked halves are the exact
// fp16 subnormals n * 2^-24 * 8^j (pn3t, j = position of the pair) or n * 2^-24 * 16^j (pn4t)
// -- an mma A register, no bias, no conversion. The 8^-j (16^-j) factor and a power of two
// 2^sigma (chosen per CTA and activation row so that any finite x fits fp16) are folded into
// the B operand: x is split into fp16 hi + lo parts (~22 bits), one mma column each (M rows
// use 2M columns, NT = ceil(2M/8) n8 tiles). The zero point is applied per block as
// d * (sum n x - z * sum x) with the per-block sums of x precomputed next to the fragments.
// Within a block the k order is free (x is permuted the same way), which lets 2-byte aligned
// words be read as aligned words pairing the high half of word i-1 with the low half of word i.
//
// Reduction. The warps' partial sums of a pass meet in shared memory; with S > 1 the
// cluster's CTAs exchange partial rows through distributed shared memory (ready / consumed
// mbarrier handshakes, double-buffered by pass) and sum them in rank order: deterministic,
// no atomics, no global scratch.
//
// Launch. Programmatic dependent launch: every CTA lets the next grid in the stream begin
// launching, and reads nothing the previous grid may write before that grid has completed
// (with the static-weights flag only the weights, which the caller declares unchanged). All
// mbarrier waits are bounded in time and report to the library's device error word.
#include <cuda.h>

#include "pnq_device.cuh"
#include "pnq_internal.h"

#include <algorithm>
#include <cstdlib>
#include <cstring>

namespace pnq {
namespace {

constexpr int kMaxM = 16;
constexpr int kTP = 4;                           // 16-row tiles per pass
constexpr int kRows = 16 * kTP;                  // rows per pass
constexpr int kColBlocks = 8;                    // blocks per tensor-map column (272 bytes of a row)
constexpr int kColBytes = kColBlocks * kBlockBytes;
constexpr int kColU32 = kColBytes / 4;           // 68 elements of the u32 tensor map
constexpr int kCols = 2;                         // columns per stage: 16 blocks
constexpr int kBoxBytes = kRows * kColBytes;     // 17408: one 64-row column box
constexpr int kTileBoxBytes = 16 * kColBytes;    // 4352: one 16-row column box
constexpr int kStageBytes = kCols * kBoxBytes;   // 34816

__host__ __device__ constexpr uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

struct PnArgs {
    CUtensorMap map_pass;  // weights as u32 [N][row_bytes / 4], box {68, 64}
    CUtensorMap map_tile;  // same tensor, box {68, 16}
    const float* X;        // [M][K]
    float* Y;              // [M][N]
    int* err;
    int N;
    int K;
    int units;             // 8-block units per row
    int M;
    int S;                 // cluster size along K
    int NS;                // stages
    int flags;             // kStaticWeights
};

enum ArgFlags : int { kStaticWeights = 1 };

// Shared-memory map (offsets from a 1024-byte aligned base), identical on host and device.
struct PnLayout {
    uint32_t bar_off;     // full[NS], empty[NS], x_ready, x_free, red_full[2], red_free[2]
    uint32_t misc_off;    // maxbits[16] u32, sig_in[16] f32, sig_out[16] f32, issued u32
    uint32_t red_off;     // [RW][kTP][NT][32 lanes][4] f32: warps' partial sums of a pass
    uint32_t part_off;    // [2][kRows][M] f32: partial rows exchanged in the cluster (S > 1)
    uint32_t z_off;       // [block][2M] f32: z * (sum of the block's scaled x, per mma column)
    uint32_t bfrag_off;   // B fragments, bfrag_unit bytes per block
    uint32_t bfrag_unit;
    uint32_t zero_off;    // 64 zero bytes read by lanes whose mma column is unused
    uint32_t stage_off;   // NS stages of kStageBytes
    uint32_t x_stage;     // x is staged in stages [x_stage, NS) at start (0: does not fit)
    uint32_t total;       // bytes from the aligned base
};

__host__ __device__ inline PnLayout make_pn_layout(int steps, int blk, int M, int NT, int RW, int units_max, int NS,
                                                   int S) {
    PnLayout L{};
    const uint32_t blocks_max = 8u * units_max;
    L.bar_off = 0;
    L.misc_off = align_up(8u * (2 * NS + 6), 16);
    L.red_off = L.misc_off + 256;
    L.part_off = align_up(L.red_off + 512u * RW * kTP * NT, 16);
    L.z_off = align_up(L.part_off + ((S > 1) ? 2u * 4u * kRows * M : 0u), 16);
    L.bfrag_off = align_up(L.z_off + blocks_max * 8u * M, 128);
    L.bfrag_unit = 64u * M * steps;  // 8M lanes x steps x 8 bytes
    L.zero_off = align_up(L.bfrag_off + L.bfrag_unit * blocks_max, 128);
    L.stage_off = align_up(L.zero_off + 64u, 1024);
    const uint32_t xbytes = static_cast<uint32_t>(M) * blocks_max * blk * 4u;
    const uint32_t xst = (xbytes + kStageBytes - 1) / kStageBytes;
    L.x_stage = (xst >= static_cast<uint32_t>(NS)) ? 0u : NS - xst;
    L.total = L.stage_off + kStageBytes * NS;
    return L;
}

// ---- decode -----------------------------------------------------------------------------

// Pair j of a (possibly re-paired) word as the f16x2 of exact subnormals (n_lo, n_hi) * 2^-24 *
// base^jj, base = 8 (pn3t) or 16 (pn4t); jj is the pair's slot after the shift that brings it
// below the fp16 exponent field.
template <int TYPE, int J>
__device__ __forceinline__ uint32_t pn_code_pair(uint32_t w) {
    if (TYPE == kTypePn3t) {
        constexpr int jj = (J < 3) ? J : J - 3;
        const uint32_t src = (J < 3) ? w : (w >> 9);
        return src & (0x00070007u << (3 * jj));
    } else {
        constexpr int jj = J & 1;
        const uint32_t src = (J < 2) ? w : (w >> 8);
        return src & (0x000F000Fu << (4 * jj));
    }
}

// 2^-(BITS * jj) for pair j: the factor folded into step j's B operand.
template <int TYPE>
__host__ __device__ constexpr float step_scale(int j) {
    return (TYPE == kTypePn3t) ? ((j % 3 == 0) ? 1.0f : (j % 3 == 1) ? 0.125f : 0.015625f)
                               : ((j & 1) ? 0.0625f : 1.0f);
}

// Element (within a block) of the low (hi_half = 0) or high code of pair j of decode word i,
// for a block starting on a 4-byte boundary (even block) or not (odd block). Odd block: natural
// word i. Even block: the aligned word at byte 4i holds the high half of word i-1 and the low
// half of word i; decode word 0 pairs the low half of word 0 with the high half of word 7.
__device__ __forceinline__ int pn_elem(int cpw, int odd_block, int i, int j, int hi_half) {
    if (odd_block) return cpw * i + 2 * j + hi_half;
    if (i == 0) return hi_half ? cpw * 7 + 2 * j + 1 : 2 * j;
    return hi_half ? cpw * i + 2 * j : cpw * (i - 1) + 2 * j + 1;
}

__device__ __forceinline__ __half split_part(float xs, int part) {
    const __half hi = __float2half_rn(xs);
    if (part == 0) return hi;
    return __float2half_rn(xs - __half2float(hi));
}

// Per-m power-of-two scaling: sigma chosen so max|x| * 2^sigma lies in [2^14, 2^15) over the
// CTA's slice (an all-zero or non-finite slice keeps sigma = 0). sig_out = 2^(24 - sigma)
// undoes both sigma and the 2^-24 of the subnormal decode.
__device__ void compute_sigma(int M, const float* xs, int klen, uint8_t* misc_p, int nct) {
    uint32_t* maxbits = reinterpret_cast<uint32_t*>(misc_p);
    float* sig_in = reinterpret_cast<float*>(misc_p + 64);
    float* sig_out = reinterpret_cast<float*>(misc_p + 128);
    const int tid = threadIdx.x;
    const uint4* xv = reinterpret_cast<const uint4*>(xs);
    const int nvec = klen / 4;  // klen is a multiple of 512
    for (int m = 0; m < M; ++m) {
        uint32_t mx = 0;
        for (int i = tid; i < nvec; i += nct) {
            const uint4 v = xv[m * nvec + i];
            mx = max(mx, max(max(v.x & 0x7FFFFFFFu, v.y & 0x7FFFFFFFu), max(v.z & 0x7FFFFFFFu, v.w & 0x7FFFFFFFu)));
        }
        mx = __reduce_max_sync(0xffffffffu, mx);
        if ((tid & 31) == 0) atomicMax(&maxbits[m], mx);
    }
    named_sync(1, nct);
    if (tid < M) {
        const uint32_t bits = maxbits[tid];
        const int E = static_cast<int>(bits >> 23);
        int sg = (bits == 0 || E >= 255) ? 0 : 141 - E;  // max < 2^(E-126)
        sg = min(100, max(-100, sg));
        sig_in[tid] = exp2i(sg);
        sig_out[tid] = exp2i(24 - sg);
    }
    named_sync(1, nct);
}

// B fragments of one block: for each n8 tile t, lanes 0..LU-1 (LU = lanes whose column is in
// use) hold 2 registers per step; steps are grouped in pairs as 16-byte records [pair][lane],
// an odd last step as 8-byte records [lane].
__device__ __forceinline__ uint32_t bfrag_offset(const PnLayout& L, int M, int steps, int blk, int t, int l, int st,
                                                 int r) {
    const int LU = min(32, 8 * M - 32 * t);
    uint32_t off = L.bfrag_off + blk * L.bfrag_unit + t * (256 * steps);
    if ((steps & 1) && st == steps - 1)
        off += (steps >> 1) * LU * 16 + l * 8 + r * 4;
    else
        off += (st >> 1) * LU * 16 + l * 16 + (st & 1) * 8 + r * 4;
    return off;
}

template <int TYPE>
__device__ void fill_fragments(int M, int nblocks, const float* xs, uint8_t* smem, const PnLayout& L, int nct) {
    using F = PnFmt<TYPE>;
    constexpr int STEPS = F::PAIRS;
    const float* sig_in = reinterpret_cast<const float*>(smem + L.misc_off + 64);
    const int klen = nblocks * F::BLK;
    const int lanes = 8 * M;
    // B fragments: one item per (pair of blocks, lane record); the block parity is unrolled
    for (int idx = threadIdx.x; idx < (nblocks / 2) * lanes; idx += nct) {
        const int bp = idx / lanes;
        const int lr = idx - bp * lanes;
        const int t = lr >> 5, l = lr & 31;
        const int g = l >> 2, tig = l & 3;
        const int col = 8 * t + g, m = col >> 1, part = col & 1;
        const float si = sig_in[m];
#pragma unroll
        for (int odd = 0; odd < 2; ++odd) {
            const int b = 2 * bp + odd;  // slices start on a multiple of 8 blocks
            const float* xb = xs + m * klen + b * F::BLK;
#pragma unroll
            for (int st = 0; st < STEPS; ++st) {
                const float sc = si * step_scale<TYPE>(st);
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int i = tig + 4 * r;
                    const __half v0 = split_part(xb[pn_elem(F::CPW, odd, i, st, 0)] * sc, part);
                    const __half v1 = split_part(xb[pn_elem(F::CPW, odd, i, st, 1)] * sc, part);
                    *reinterpret_cast<uint32_t*>(smem + bfrag_offset(L, M, STEPS, b, t, l, st, r)) =
                        pack_half2(v0, v1);
                }
            }
        }
    }
    // z * sum over the block of what the decoded A multiplies (2^-24 * base^jj * B element):
    // one warp per block, lanes over the block's elements, then a shuffle reduction
    float* z = reinterpret_cast<float*>(smem + L.z_off);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = nct >> 5;
    for (int b = warp; b < nblocks; b += nwarps) {
        for (int m = 0; m < M; ++m) {
            const float* xb = xs + m * klen + b * F::BLK;
            const float si = sig_in[m];
            float shi = 0.0f, slo = 0.0f;
            for (int e = lane; e < F::BLK; e += 32) {
                const float sc = step_scale<TYPE>((e % F::CPW) >> 1);
                const float v = xb[e] * (si * sc);
                const __half h = __float2half_rn(v);
                const float hf = __half2float(h);
                const float lf = __half2float(__float2half_rn(v - hf));
                const float f = 5.9604644775390625e-08f / sc;  // 2^-24 * base^jj
                shi = fmaf(f, hf, shi);
                slo = fmaf(f, lf, slo);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                shi += __shfl_xor_sync(0xffffffffu, shi, o);
                slo += __shfl_xor_sync(0xffffffffu, slo, o);
            }
            if (lane == 0) {
                z[b * 2 * M + 2 * m] = static_cast<float>(F::Z) * shi;
                z[b * 2 * M + 2 * m + 1] = static_cast<float>(F::Z) * slo;
            }
        }
    }
}

// One block (ODD: starts 2 bytes past a 4-byte boundary) for the first `tiles` of kTP tiles:
// rowp[tile][0] = row g, [1] = row g + 8 (stage addresses of the block's column).
template <int TYPE, int NT, int ODD, bool FULL>
__device__ __forceinline__ void pn_block(const uint8_t* const (&rowp)[kTP][2], int off, const uint8_t* bblk,
                                         const float* zblk, const uint8_t* zero, int M, int lane, int tiles,
                                         float (&acc)[kTP][NT][4]) {
    using F = PnFmt<TYPE>;
    constexpr int STEPS = F::PAIRS;
    const int tig = lane & 3;
    float d[kTP][2];
    uint32_t wa[kTP][2], wb[kTP][2];
#pragma unroll
    for (int tp = 0; tp < kTP; ++tp) {
        if (FULL || tp < tiles) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint8_t* p = rowp[tp][h] + off;
                d[tp][h] = __half2float(*reinterpret_cast<const __half*>(p));
                if (ODD) {
                    wa[tp][h] = *reinterpret_cast<const uint32_t*>(p + 2 + 4 * tig);
                    wb[tp][h] = *reinterpret_cast<const uint32_t*>(p + 18 + 4 * tig);
                } else {
                    const uint32_t w0 = *reinterpret_cast<const uint32_t*>(p + 4 * tig);
                    wb[tp][h] = *reinterpret_cast<const uint32_t*>(p + 16 + 4 * tig);
                    const uint32_t x8 = *reinterpret_cast<const uint32_t*>(p + 32);
                    const uint32_t pr = prmt(w0, x8, 0x5432u);
                    wa[tp][h] = (tig == 0) ? pr : w0;
                }
            }
        }
    }
    // B registers and zero-point corrections for this lane's columns (unused columns read zeros)
    uint32_t b[NT][STEPS][2];
    float zh[NT], zl[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const int LU = min(32, 8 * M - 32 * t);
        const bool live = lane < LU;
        const uint8_t* base = bblk + t * (256 * STEPS);
#pragma unroll
        for (int q = 0; q < STEPS / 2; ++q) {
            const uint4 v = *reinterpret_cast<const uint4*>(live ? base + q * LU * 16 + lane * 16 : zero);
            b[t][2 * q][0] = v.x;
            b[t][2 * q][1] = v.y;
            b[t][2 * q + 1][0] = v.z;
            b[t][2 * q + 1][1] = v.w;
        }
        if (STEPS & 1) {
            const uint2 v = *reinterpret_cast<const uint2*>(live ? base + (STEPS / 2) * LU * 16 + lane * 8 : zero);
            b[t][STEPS - 1][0] = v.x;
            b[t][STEPS - 1][1] = v.y;
        }
        const int m = 4 * t + tig;
        const float2 zz = *reinterpret_cast<const float2*>(m < M ? reinterpret_cast<const uint8_t*>(zblk + 2 * m) : zero);
        zh[t] = zz.x;
        zl[t] = zz.y;
    }
    float c[kTP][NT][4];
#define PNQ_STEP(J)                                                                                           \
    {                                                                                                         \
        _Pragma("unroll") for (int tp = 0; tp < kTP; ++tp) {                                                  \
            if (FULL || tp < tiles) {                                                                         \
                const uint32_t a0 = pn_code_pair<TYPE, J>(wa[tp][0]), a1 = pn_code_pair<TYPE, J>(wa[tp][1]);  \
                const uint32_t a2 = pn_code_pair<TYPE, J>(wb[tp][0]), a3 = pn_code_pair<TYPE, J>(wb[tp][1]);  \
                _Pragma("unroll") for (int t = 0; t < NT; ++t) {                                              \
                    if (J == 0)                                                                               \
                        mma_f16_16816_z(c[tp][t], a0, a1, a2, a3, b[t][J][0], b[t][J][1]);                     \
                    else                                                                                      \
                        mma_f16_16816(c[tp][t], a0, a1, a2, a3, b[t][J][0], b[t][J][1]);                       \
                }                                                                                             \
            }                                                                                                 \
        }                                                                                                     \
    }
    PNQ_STEP(0)
    PNQ_STEP(1)
    PNQ_STEP(2)
    PNQ_STEP(3)
    if constexpr (STEPS == 5) PNQ_STEP(4)
#undef PNQ_STEP
#pragma unroll
    for (int tp = 0; tp < kTP; ++tp) {
        if (FULL || tp < tiles) {
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                acc[tp][t][0] = fmaf(d[tp][0], c[tp][t][0] - zh[t], acc[tp][t][0]);
                acc[tp][t][1] = fmaf(d[tp][0], c[tp][t][1] - zl[t], acc[tp][t][1]);
                acc[tp][t][2] = fmaf(d[tp][1], c[tp][t][2] - zh[t], acc[tp][t][2]);
                acc[tp][t][3] = fmaf(d[tp][1], c[tp][t][3] - zl[t], acc[tp][t][3]);
            }
        }
    }
}

// ---- the kernel ---------------------------------------------------------------------------------

template <int TYPE, int NT, int kRW>
__global__ void __launch_bounds__(32 * (kRW + 1), 1) pn_gemv_kernel(const __grid_constant__ PnArgs a) {
    using F = PnFmt<TYPE>;
    constexpr int STEPS = F::PAIRS;
    constexpr int kBlkPerWarp = kCols * kColBlocks / kRW;  // blocks of a stage per consumer warp (even)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const uint32_t rank = (a.S > 1) ? cluster_ctarank() : 0u;
    const int units_max = (a.units + a.S - 1) / a.S;
    const PnLayout L = make_pn_layout(STEPS, F::BLK, a.M, NT, kRW, units_max, a.NS, a.S);
    // this CTA's K slice, in 8-block units
    const int u0 = static_cast<int>((static_cast<int64_t>(rank) * a.units) / a.S);
    const int nunits = static_cast<int>((static_cast<int64_t>(rank + 1) * a.units) / a.S) - u0;
    const int nchunks = (nunits + kCols - 1) / kCols;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // this cluster's tiles: a balanced contiguous share of the 16-row tiles
    const int T16 = (a.N + 15) / 16;
    const int cl = blockIdx.y, ncl = gridDim.y;
    const int t_begin = static_cast<int>((static_cast<int64_t>(cl) * T16) / ncl);
    const int t_end = static_cast<int>((static_cast<int64_t>(cl + 1) * T16) / ncl);
    const int npasses = (t_end - t_begin + kTP - 1) / kTP;
    const int total_chunks = npasses * nchunks;

    const uint32_t bar0 = smem_addr(smem + L.bar_off);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (a.NS + s); };
    const uint32_t x_ready = bar0 + 8u * (2 * a.NS);
    const uint32_t x_free = bar0 + 8u * (2 * a.NS + 1);
    auto red_full = [&](int b) { return bar0 + 8u * (2 * a.NS + 2 + b); };
    auto red_free = [&](int b) { return bar0 + 8u * (2 * a.NS + 4 + b); };
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L.misc_off);
    float* xs = reinterpret_cast<float*>(smem + L.stage_off + L.x_stage * kStageBytes);

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.NS; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), kRW);
        }
        mbar_init(x_ready, 1);
        mbar_init(x_free, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(red_full(b), a.S);
            mbar_init(red_free(b), a.S);
        }
        mbar_fence_init();
        griddep_launch_dependents();
    }
    if (threadIdx.x < 16) {
        misc[threadIdx.x] = 0u;                                                // maxbits
        reinterpret_cast<uint32_t*>(smem + L.zero_off)[threadIdx.x] = 0u;      // zero area
    }
    if (threadIdx.x == 16) misc[48] = 0u;  // issued
    __syncthreads();
    if (a.S > 1) cluster_sync();  // every CTA's barriers exist before any remote arrive

    if (warp == kRW) {
        // ---------------- producer warp ----------------
        const uint64_t pol = l2_policy_evict_first();
        bool ok = true;
        auto issue = [&](int gch) {
            const int p = gch / nchunks, c = gch - p * nchunks;
            const int s = gch % a.NS;
            if (gch >= a.NS) {
                if (!mbar_wait_bounded(empty_bar(s), ((gch / a.NS) - 1) & 1)) return false;
            } else if (s >= static_cast<int>(L.x_stage)) {
                if (!mbar_wait_bounded(x_free, 0)) return false;
            }
            if (lane == 0) {
                const int t0 = t_begin + p * kTP;
                const int tiles = min(kTP, t_end - t0);
                const int ncol = min(kCols, nunits - c * kCols);
                const uint32_t dst = smem_addr(smem + L.stage_off + s * kStageBytes);
                if (tiles == kTP) {
                    mbar_arrive_expect_tx(full_bar(s), static_cast<uint32_t>(ncol * kBoxBytes));
                    for (int h = 0; h < ncol; ++h)
                        tma_load_2d(dst + h * kBoxBytes, &a.map_pass, (u0 + c * kCols + h) * kColU32, 16 * t0, full_bar(s),
                                    pol);
                } else {
                    mbar_arrive_expect_tx(full_bar(s), static_cast<uint32_t>(ncol * tiles * kTileBoxBytes));
                    for (int h = 0; h < ncol; ++h)
                        for (int t = 0; t < tiles; ++t)
                            tma_load_2d(dst + h * kBoxBytes + t * kTileBoxBytes, &a.map_tile,
                                        (u0 + c * kCols + h) * kColU32, 16 * (t0 + t), full_bar(s), pol);
                }
            }
            __syncwarp();
            return true;
        };
        int gch = 0;
        if (a.flags & kStaticWeights) {
            // weights are declared unchanged by earlier work: stream them into the stages that do
            // not hold x before the previous grid in the stream has finished
            for (; ok && gch < min(total_chunks, static_cast<int>(L.x_stage)); ++gch) ok = issue(gch);
        }
        griddep_wait();
        {
            // the CTA's slice of x: one bulk copy per activation row (16-byte aligned: X is, and the
            // slice starts at a multiple of 512 elements)
            const uint32_t xbytes = static_cast<uint32_t>(nunits * kColBlocks * F::BLK * 4);
            if (lane == 0) mbar_arrive_expect_tx(x_ready, xbytes * a.M);
            __syncwarp();
            const float* xsrc = a.X + static_cast<size_t>(u0) * kColBlocks * F::BLK;
            if (lane < a.M)
                bulk_g2s_plain(smem_addr(xs) + lane * xbytes, xsrc + static_cast<size_t>(lane) * a.K, xbytes, x_ready);
        }
        for (; ok && gch < total_chunks; ++gch) ok = issue(gch);
        if (!ok && lane == 0) record_error(a.err, kErrEmptyWait);
        if (lane == 0) misc[48] = static_cast<uint32_t>(ok ? total_chunks : gch);
    } else {
        // ---------------- consumer warps ----------------
        constexpr int nct = 32 * kRW;
        const int nblocks = nunits * kColBlocks;
        if (!mbar_wait_bounded(x_ready, 0) && lane == 0) record_error(a.err, kErrFullWait);
        compute_sigma(a.M, xs, nblocks * F::BLK, smem + L.misc_off, nct);
        fill_fragments<TYPE>(a.M, nblocks, xs, smem, L, nct);
        named_sync(1, nct);
        if (threadIdx.x == 0) mbar_arrive(x_free);  // the x stages may now take weights

        const int g = lane >> 2, tig = lane & 3;
        const float* sig_out = reinterpret_cast<const float*>(smem + L.misc_off + 128);
        const uint8_t* zero = smem + L.zero_off;
        const float* zarr = reinterpret_cast<const float*>(smem + L.z_off);
        float* red = reinterpret_cast<float*>(smem + L.red_off);
        const uint32_t part_addr = smem_addr(smem + L.part_off);
        const uint32_t part_stride = 4u * kRows * a.M;  // bytes per pass buffer
        const int hcol = (warp * kBlkPerWarp) / kColBlocks;  // the stage column this warp reads
        const int cblk = (warp * kBlkPerWarp) % kColBlocks;  // its first block within the column
        bool ok = true;
        int p = 0;
        for (; p < npasses && ok; ++p) {
            const int t0 = t_begin + p * kTP;
            const int tiles = min(kTP, t_end - t0);
            const int rbase = 16 * t0;
            float acc[kTP][NT][4];
#pragma unroll
            for (int tp = 0; tp < kTP; ++tp)
#pragma unroll
                for (int t = 0; t < NT; ++t) acc[tp][t][0] = acc[tp][t][1] = acc[tp][t][2] = acc[tp][t][3] = 0.0f;
            for (int c = 0; c < nchunks; ++c) {
                const int gch = p * nchunks + c;
                const int s = gch % a.NS;
                if (!mbar_wait_bounded(full_bar(s), (gch / a.NS) & 1)) {
                    if (lane == 0) record_error(a.err, kErrFullWait);
                    ok = false;
                    break;
                }
                if (c * kCols + hcol < nunits) {
                    const uint8_t* colp = smem + L.stage_off + s * kStageBytes + hcol * kBoxBytes;
                    const uint8_t* rowp[kTP][2];
#pragma unroll
                    for (int tp = 0; tp < kTP; ++tp) {
                        rowp[tp][0] = colp + (16 * tp + g) * kColBytes;
                        rowp[tp][1] = rowp[tp][0] + 8 * kColBytes;
                    }
#pragma unroll
                    for (int j = 0; j < kBlkPerWarp; j += 2) {
                        const int blk = (c * kCols + hcol) * kColBlocks + cblk + j;  // block index in the slice
                        const uint8_t* b0 = smem + L.bfrag_off + blk * L.bfrag_unit;
                        const float* z0 = zarr + blk * 2 * a.M;
                        const int off = kBlockBytes * (cblk + j);
                        if (tiles == kTP) {
                            pn_block<TYPE, NT, 0, true>(rowp, off, b0, z0, zero, a.M, lane, tiles, acc);
                            pn_block<TYPE, NT, 1, true>(rowp, off + kBlockBytes, b0 + L.bfrag_unit, z0 + 2 * a.M, zero,
                                                        a.M, lane, tiles, acc);
                        } else {
                            pn_block<TYPE, NT, 0, false>(rowp, off, b0, z0, zero, a.M, lane, tiles, acc);
                            pn_block<TYPE, NT, 1, false>(rowp, off + kBlockBytes, b0 + L.bfrag_unit, z0 + 2 * a.M, zero,
                                                         a.M, lane, tiles, acc);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty_bar(s));
            }
            if (!ok) break;

            // ---- reduce the warps' K shares, then (S > 1) the cluster's K slices
            const int b = p & 1;
#pragma unroll
            for (int tp = 0; tp < kTP; ++tp)
                if (tp < tiles)
#pragma unroll
                    for (int t = 0; t < NT; ++t)
                        *reinterpret_cast<float4*>(red + ((((warp * kTP + tp) * NT + t) * 32 + lane) * 4)) =
                            make_float4(acc[tp][t][0], acc[tp][t][1], acc[tp][t][2], acc[tp][t][3]);
            if (a.S > 1 && p >= 2 && !mbar_wait_cluster_bounded(red_free(b), ((p - 2) >> 1) & 1)) {
                if (lane == 0) record_error(a.err, kErrReduceWait);
                ok = false;
            }
            named_sync(1, nct);
            if (warp < tiles) {
                float sum[NT][4];
#pragma unroll
                for (int t = 0; t < NT; ++t) sum[t][0] = sum[t][1] = sum[t][2] = sum[t][3] = 0.0f;
#pragma unroll
                for (int w = 0; w < kRW; ++w)
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        const float4 v = *reinterpret_cast<const float4*>(red + ((((w * kTP + warp) * NT + t) * 32 + lane) * 4));
                        sum[t][0] += v.x;
                        sum[t][1] += v.y;
                        sum[t][2] += v.z;
                        sum[t][3] += v.w;
                    }
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const int m = 4 * t + tig;
                    if (m < a.M) {
                        const float so = sig_out[m];
                        const float y0 = (sum[t][0] + sum[t][1]) * so;
                        const float y1 = (sum[t][2] + sum[t][3]) * so;
                        const int ra = 16 * warp + g, rb = ra + 8;
                        if (a.S == 1) {
                            if (rbase + ra < a.N) a.Y[static_cast<size_t>(m) * a.N + rbase + ra] = y0;
                            if (rbase + rb < a.N) a.Y[static_cast<size_t>(m) * a.N + rbase + rb] = y1;
                        } else {
                            float* part = reinterpret_cast<float*>(smem + L.part_off + b * part_stride);
                            part[ra * a.M + m] = y0;
                            part[rb * a.M + m] = y1;
                        }
                    }
                }
            }
            named_sync(1, nct);
            if (a.S > 1) {
                // this CTA's partial rows of the pass are complete: tell every rank
                if (threadIdx.x == 0) {
                    fence_acq_rel_cluster();
                    for (int q = 0; q < a.S; ++q) mbar_arrive_remote(mapa_shared(red_full(b), q));
                }
                if (!mbar_wait_cluster_bounded(red_full(b), (p >> 1) & 1)) {
                    if (lane == 0) record_error(a.err, kErrReduceWait);
                    ok = false;
                }
                // rank r finishes the tiles t with t % S == r: sum the S partials in rank order
                const uint32_t pb = part_addr + b * part_stride;
                for (int idx = threadIdx.x; idx < tiles * 16 * a.M; idx += nct) {
                    const int rr = idx / a.M, m = idx - rr * a.M;
                    if (((rr >> 4) % a.S) != static_cast<int>(rank) || rbase + rr >= a.N) continue;
                    float sum = 0.0f;
                    for (int q = 0; q < a.S; ++q) sum += ld_dsmem_f32_at(mapa_shared(pb + 4u * idx, q));
                    a.Y[static_cast<size_t>(m) * a.N + rbase + rr] = sum;
                }
                named_sync(1, nct);
                if (threadIdx.x == 0) {
                    fence_acq_rel_cluster();
                    for (int q = 0; q < a.S; ++q) mbar_arrive_remote(mapa_shared(red_free(b), q));
                }
            }
        }
        if (a.S > 1) {
            // every rank has finished reading this CTA's last partial buffers
            for (int q = max(0, p - 2); q < p; ++q)
                if (!mbar_wait_cluster_bounded(red_free(q & 1), (q >> 1) & 1) && lane == 0)
                    record_error(a.err, kErrReduceWait);
        }
    }

    __syncthreads();
    // Drain: no CTA leaves while a copy it issued may still be writing its shared memory.
    if (warp == kRW && lane == 0) {
        if (!mbar_wait_bounded(x_ready, 0)) record_error(a.err, kErrDrainWait);
        const int issued = static_cast<int>(misc[48]);
        for (int c = max(0, issued - a.NS); c < issued; ++c)
            if (!mbar_wait_bounded(full_bar(c % a.NS), (c / a.NS) & 1)) record_error(a.err, kErrDrainWait);
    }
    if (a.S > 1) cluster_sync();  // no CTA leaves while a peer may still address its shared memory
}

// ---- host side --------------------------------------------------------------------------------------

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn tensor_map_encoder() {
    static EncodeFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeFn>(nullptr);
        return reinterpret_cast<EncodeFn>(p);
    }();
    return fn;
}

// Weights viewed as u32 [N][row_bytes / 4]; box {68, rows}. Rows past N read as zeros.
bool encode_weight_map(CUtensorMap* map, const uint8_t* W, int64_t N, int64_t row_bytes, int box_rows) {
    EncodeFn enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes / 4), static_cast<cuuint64_t>(N)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kColU32), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint8_t*>(W), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int TYPE, int NT, int kRW>
cudaError_t prepare_kernel(int S, size_t smem_bytes) {
    auto kern = pn_gemv_kernel<TYPE, NT, kRW>;
    // raised once per device and size (so never while a stream is being captured after the first
    // eager call)
    static size_t opted[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (opted[dev] < smem_bytes) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_bytes));
        if (e != cudaSuccess) return e;
        opted[dev] = smem_bytes;
    }
    (void)S;
    return cudaSuccess;
}

// Co-resident clusters of S CTAs with this shared-memory size (cached per device, S, size).
template <int TYPE, int NT, int kRW>
int resident_clusters(int S, size_t smem_bytes) {
    struct Entry { int dev, S; size_t smem; int n; };
    static Entry cache[64];
    static int used = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    for (int i = 0; i < used; ++i)
        if (cache[i].dev == dev && cache[i].S == S && cache[i].smem == smem_bytes) return cache[i].n;
    if (prepare_kernel<TYPE, NT, kRW>(S, smem_bytes) != cudaSuccess) return 0;
    auto kern = pn_gemv_kernel<TYPE, NT, kRW>;
    int n = 0;
    if (S == 1) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32 * (kRW + 1), smem_bytes) != cudaSuccess)
            return 0;
        n = per_sm * device_sm_count();
    } else {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(S, 1024, 1);
        cfg.blockDim = dim3(32 * (kRW + 1), 1, 1);
        cfg.dynamicSmemBytes = smem_bytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = S;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
    }
    if (used < 64) cache[used++] = Entry{dev, S, smem_bytes, n};
    return n;
}

// Environment override "rw,S,_,ns" (fields 0 = automatic; rw is ignored here), read once.
MmaConfig env_config() {
    static MmaConfig cfg = [] {
        MmaConfig c{0, 0, 0, 0};
        if (const char* s = std::getenv("PNQ_GEMV_CFG")) {
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

template <int TYPE, int NT, int kRW>
cudaError_t plan_and_launch(PnArgs& a, const MmaConfig& cfg, cudaStream_t stream) {
    using F = PnFmt<TYPE>;
    const int U = a.units;
    const int T16 = (a.N + 15) / 16;
    auto layout_for = [&](int S, int ns) {
        return make_pn_layout(F::PAIRS, F::BLK, a.M, NT, kRW, (U + S - 1) / S, ns, S);
    };
    auto fits = [&](const PnLayout& L) { return L.total + 1024u <= 227u * 1024u && L.x_stage >= 1; };
    auto stages_for = [&](int S) {
        if (cfg.ns > 0) return fits(layout_for(S, cfg.ns)) ? cfg.ns : 0;
        for (int ns = 4; ns >= 3; --ns)
            if (fits(layout_for(S, ns))) return ns;
        for (int ns = 5; ns <= 6; ++ns)  // x may need more stages than the default
            if (fits(layout_for(S, ns))) return ns;
        return 0;
    };
    const int s_list[] = {1, 2, 4, 8};
    int s_forced = 0;  // a requested cluster size, rounded down to the list and to U
    if (cfg.S > 0)
        for (int S : s_list)
            if (S <= std::min(cfg.S, U)) s_forced = S;
    int best_S = 0, best_ns = 0, best_clusters = 0;
    int64_t best_cost = INT64_MAX;
    for (int S : s_list) {
        if (S > U) break;
        if (s_forced > 0 && S != s_forced) continue;
        const int ns = stages_for(S);
        if (ns == 0) continue;
        const int resident = resident_clusters<TYPE, NT, kRW>(S, layout_for(S, ns).total + 1024u);
        if (resident < 1) continue;
        const int clusters = std::min(resident, T16);
        // makespan of the busiest CTA in (16-row tile x 8-block unit) items, plus per-pass costs
        const int64_t tiles = (T16 + clusters - 1) / clusters;
        const int64_t units = (U + S - 1) / S;
        const int64_t cost = tiles * units * 8 + ((tiles + kTP - 1) / kTP) * (S > 1 ? 40 : 16) + units * 4;
        if (cost < best_cost) {
            best_cost = cost;
            best_S = S;
            best_ns = ns;
            best_clusters = clusters;
        }
    }
    if (best_S == 0) return cudaErrorNotSupported;
    a.S = best_S;
    a.NS = best_ns;
    const size_t smem_bytes = layout_for(best_S, best_ns).total + 1024u;
    cudaError_t e = prepare_kernel<TYPE, NT, kRW>(a.S, smem_bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(a.S, best_clusters, 1);
    lc.blockDim = dim3(32 * (kRW + 1), 1, 1);
    lc.dynamicSmemBytes = smem_bytes;
    lc.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (a.S > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = a.S;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    // may begin while the previous grid in the stream finishes (see griddep_wait in the kernel)
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    lc.attrs = attr;
    lc.numAttrs = n;
    return cudaLaunchKernelEx(&lc, pn_gemv_kernel<TYPE, NT, kRW>, a);
}

template <int TYPE>
cudaError_t launch_typed(PnArgs& a, const MmaConfig& cfg, cudaStream_t stream) {
    const int nt = (2 * a.M + 7) / 8;
    // eight consumer warps while the registers allow it (one tile of n8 columns), four otherwise
    if (nt <= 1) return plan_and_launch<TYPE, 1, 8>(a, cfg, stream);
    if (nt <= 2) return plan_and_launch<TYPE, 2, 4>(a, cfg, stream);
    return plan_and_launch<TYPE, 4, 4>(a, cfg, stream);
}

}  // namespace

cudaError_t launch_pn_gemv_mma(int type, const uint8_t* W, int64_t N, int64_t K, const float* X, int M, float* Y,
                               int* err, MmaConfig cfg, bool static_weights, cudaStream_t stream) {
    if (N == 0) return cudaSuccess;
    const int blk = (type == kTypePn3t) ? 80 : 64;
    const int64_t nb = K / blk;
    if (N > INT32_MAX || nb % 8 != 0 || nb / 8 > INT32_MAX / 2 || M < 1 || M > kMaxM) return cudaErrorNotSupported;
    if (reinterpret_cast<uintptr_t>(W) % 16 != 0 || reinterpret_cast<uintptr_t>(X) % 16 != 0)
        return cudaErrorNotSupported;
    const MmaConfig env = env_config();
    if (cfg.S <= 0) cfg.S = env.S;
    if (cfg.ns <= 0) cfg.ns = env.ns;
    if (cfg.ns != 0 && (cfg.ns < 2 || cfg.ns > 16)) return cudaErrorInvalidValue;
    PnArgs a{};
    const int64_t row_bytes = nb * kBlockBytes;
    if (!encode_weight_map(&a.map_pass, W, N, row_bytes, kRows) || !encode_weight_map(&a.map_tile, W, N, row_bytes, 16))
        return cudaErrorNotSupported;
    a.X = X;
    a.Y = Y;
    a.err = err;
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.units = static_cast<int>(nb / 8);
    a.M = M;
    a.flags = static_weights ? kStaticWeights : 0;
    if (type == kTypePn3t) return launch_typed<kTypePn3t>(a, cfg, stream);
    return launch_typed<kTypePn4t>(a, cfg, stream);
}

}  // namespace pnq
