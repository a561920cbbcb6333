// pnq_gemv_tc.cu -- PN (pn3t / pn4t) GEMV on the fifth-generation tensor cores (tcgen05), sm_103a.
//
// Computes Y[m][n] = sum_k w[n][k] x[m][k] for 1 <= M <= 16, with w = d * (n - z) decoded in
// registers from the 34-byte blocks of the "PN weight format" page (sections Block layout and
// Value) just before the multiply.
//
// Items and schedule (stream-K). The weight matrix is cut into items of 128 rows x one K unit
// of 8 blocks (272 bytes per row). Items are numbered unit-major (item = u * T + t for row
// tile t of T) and every CTA of a persistent grid (one per SM) takes an equal contiguous share,
// so all SMs stream the same number of bytes and a CTA's items touch at most a few K units.
//
// Memory pipeline. One producer thread loads one item per stage with a 2-D tensor-map copy
// (box 272 bytes x 128 rows, L2 evict-first; rows past N read as zeros) into an NS-stage ring
// under mbarriers. At start it also copies the CTA's slice of x (fp32) into the last stages.
//
// Decode (8 warps). A thread owns one weight row = one tensor-memory lane; warps 0-3 decode
// blocks 0-3 of each unit, warps 4-7 blocks 4-7. A 32-bit word of a block holds two codes at
// the same shift in its two 16-bit halves; masking out such a pair leaves in each half the
// exact fp16 subnormal n * 2^-24 * 8^j (pn3t; 16^j for pn4t, j = position of the pair). Eight
// masked words are one K=16 slice of the A operand and go straight to tensor memory
// (tcgen05.st); a block is 5 (pn3t) or 4 (pn4t) slices. The k order inside a block is free as
// long as B uses the same order, which lets the 2-byte aligned words of even blocks be read as
// aligned words that pair the high half of word i-1 with the low half of word i.
//
// B operand (shared memory, K-major, canonical no-swizzle layout): per block and slice a
// 16 x 16 fp16 tile of x times 8^-j (16^-j) times 2^sigma, sigma chosen per CTA and activation
// row so that max|x| * 2^sigma lies in [2^14, 2^15), split into fp16 hi + lo parts (~22 bits).
// M <= 8: column 2m + p holds part p of row m, one MMA per slice. M > 8: column m, the parts in
// two tiles accumulated into the same D (two MMAs per slice).
//
// MMA (one thread): per block, D (128 x 16 f32 in tensor memory) = sum over its slices of A x B
// (tcgen05.mma kind::f16, A from tensor memory), then tcgen05.commit to an mbarrier.
//
// Epilogue. The block scale d and the zero point are applied when the decode warps read D
// back: acc += d * (D - Z), Z = z * (sum over the block of B times 2^-24 * 8^j), computed in
// fp32 beside B. Two sets of A / D columns (one per warp set) let the decode of item i+1
// overlap the MMAs of item i.
//
// Reduction. After each item the decode warps leave their row sums in shared memory; a
// reducer warp adds the two sets, writes the item's rows to a workspace slot and counts the
// item on its row tile; the CTA that brings a tile's count to U sums the tile's U slots in unit
// order (so the result does not depend on timing) and writes Y.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <type_traits>
#include <utility>

#include "pnq_device.cuh"
#include "pnq_internal.h"

namespace pnq {
namespace {

constexpr int kTileRows = 128;                         // rows per item = MMA M
constexpr int kUnitBlocks = 8;                         // blocks per K unit
constexpr int kUnitBytes = kUnitBlocks * kBlockBytes;  // 272 bytes of a row per unit
constexpr int kUnitU32 = kUnitBytes / 4;               // 68
constexpr int kStageBytes = kTileRows * kUnitBytes;    // 34816
constexpr int kSetBlocks = 4;                          // blocks per warp set and unit
constexpr int kDecodeWarps = 8;
constexpr int kProducerWarp = 8, kMmaWarp = 9, kReducerWarp = 10;
constexpr int kThreads = 32 * 11;
constexpr int kDecodeThreads = 32 * kDecodeWarps;
constexpr int kN = 16;  // MMA N: D columns per block
// instruction descriptor: D f32, A and B f16, both K-major, N = 16, M = 128
constexpr uint32_t kIdesc = (1u << 4) | (static_cast<uint32_t>(kN >> 3) << 17) |
                            (static_cast<uint32_t>(kTileRows >> 4) << 24);
constexpr int kBTile = 512;                  // one 16 x 16 fp16 B tile
constexpr uint32_t kLbo = 128, kSbo = 256;   // core-matrix strides along K / along N
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxStages = 8;
constexpr unsigned kStaticWeights = 1u;
constexpr size_t kSmemLimit = 227u * 1024u;

template <int TYPE>
struct TcShape {
    static constexpr int STEPS = PnFmt<TYPE>::PAIRS;
    static constexpr int ACOLS = kSetBlocks * 8 * STEPS;     // A columns per set
    static constexpr int SETCOLS = ACOLS + kSetBlocks * kN;  // A + D columns per set
};
static_assert(2 * TcShape<kTypePn3t>::SETCOLS <= static_cast<int>(kTmemCols), "tensor memory");
static_assert(2 * TcShape<kTypePn4t>::SETCOLS <= static_cast<int>(kTmemCols), "tensor memory");

struct TcArgs {
    CUtensorMap map;  // weights as u32 [N][row_bytes / 4], box {68, 128}
    const float* X;
    float* Y;
    float* ws;       // partial rows [T][U][M][128]
    uint32_t* cnt;   // [T] items counted per row tile (zero between launches)
    int* err;
    long long items;
    int N, K, M, T, U, NS, x_stage;
    unsigned flags;
    uint32_t bar_off, misc_off, z_off, part_off, b_off, stage_off;
};

// 2^-(BITS * jj) for slice j: the factor folded into slice j of B, and its inverse.
template <int TYPE>
__device__ __forceinline__ float step_scale(int j) {
    return (TYPE == kTypePn3t) ? ((j % 3 == 0) ? 1.0f : (j % 3 == 1) ? 0.125f : 0.015625f)
                               : ((j & 1) ? 0.0625f : 1.0f);
}
template <int TYPE>
__device__ __forceinline__ float step_scale_inv(int j) {
    return (TYPE == kTypePn3t) ? ((j % 3 == 0) ? 1.0f : (j % 3 == 1) ? 8.0f : 64.0f) : ((j & 1) ? 16.0f : 1.0f);
}

// Masked pair j of a word (w) or of the word shifted right by 9 (pn3t) / 8 (pn4t) (ws): the two
// codes at shift BITS * (j mod per-half) in the low bits of each 16-bit half.
template <int TYPE, int J>
__device__ __forceinline__ uint32_t code_pair(uint32_t w, uint32_t ws) {
    if constexpr (TYPE == kTypePn3t) {
        if constexpr (J < 3) return w & (0x00070007u << (3 * J));
        else return ws & (0x00070007u << (3 * (J - 3)));
    } else {
        if constexpr (J < 2) return w & (0x000F000Fu << (4 * J));
        else return ws & (0x000F000Fu << (4 * (J - 2)));
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

__device__ __forceinline__ __half split_part(float v, int part) {
    const __half hi = __float2half_rn(v);
    if (part == 0) return hi;
    return __float2half_rn(v - __half2float(hi));
}

// Decode block BI of warp set H from the row window (36 words = bytes 128*H .. 128*H+143 of the
// row's 272-byte unit) into tensor-memory columns a_taddr .. a_taddr + 8*STEPS - 1; returns d.
template <int TYPE, int H, int BI>
__device__ __forceinline__ float decode_block(const uint32_t (&win)[36], uint32_t a_taddr) {
    constexpr int b = kSetBlocks * H + BI;
    constexpr int off = kBlockBytes * b - 128 * H;  // byte offset of the block in the window
    constexpr int SH = (TYPE == kTypePn3t) ? 9 : 8;
    uint32_t R[8];
    uint32_t dbits;
    if constexpr ((b & 1) == 0) {
        constexpr int wi = off / 4;
        dbits = win[wi] & 0xFFFFu;
        R[0] = prmt(win[wi], win[wi + 8], 0x5432u);
#pragma unroll
        for (int i = 1; i < 8; ++i) R[i] = win[wi + i];
    } else {
        constexpr int wd = (off - 2) / 4;
        dbits = win[wd] >> 16;
#pragma unroll
        for (int i = 0; i < 8; ++i) R[i] = win[wd + 1 + i];
    }
    uint32_t S[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) S[i] = R[i] >> SH;
#define PNQ_TC_SLICE(J)                                                                                       \
    if constexpr (J < PnFmt<TYPE>::PAIRS)                                                                     \
        tmem_st8(a_taddr + 8 * (J), code_pair<TYPE, J>(R[0], S[0]), code_pair<TYPE, J>(R[1], S[1]),            \
                 code_pair<TYPE, J>(R[2], S[2]), code_pair<TYPE, J>(R[3], S[3]), code_pair<TYPE, J>(R[4], S[4]), \
                 code_pair<TYPE, J>(R[5], S[5]), code_pair<TYPE, J>(R[6], S[6]), code_pair<TYPE, J>(R[7], S[7]));
    PNQ_TC_SLICE(0)
    PNQ_TC_SLICE(1)
    PNQ_TC_SLICE(2)
    PNQ_TC_SLICE(3)
    PNQ_TC_SLICE(4)
#undef PNQ_TC_SLICE
    return __half2float(__ushort_as_half(static_cast<unsigned short>(dbits)));
}

// Shared-memory layout helpers (offsets relative to the 1024-aligned base).
struct Smem {
    uint8_t* base;
    const TcArgs* a;
    __device__ uint32_t bar(int i) const { return smem_addr(base + a->bar_off) + 8u * i; }
    __device__ uint32_t full(int s) const { return bar(s); }
    __device__ uint32_t empty(int s) const { return bar(a->NS + s); }
    __device__ uint32_t x_ready() const { return bar(2 * a->NS); }
    __device__ uint32_t x_free() const { return bar(2 * a->NS + 1); }
    // block slot (set h, block bi): A written (4 warps arrive) / its MMAs completed (commit)
    __device__ uint32_t slot_full(int h, int bi) const { return bar(2 * a->NS + 2 + h * kSetBlocks + bi); }
    __device__ uint32_t slot_done(int h, int bi) const { return bar(2 * a->NS + 10 + h * kSetBlocks + bi); }
    __device__ uint32_t part_full(int b) const { return bar(2 * a->NS + 18 + b); }
    __device__ uint32_t part_free(int b) const { return bar(2 * a->NS + 20 + b); }
    __device__ uint32_t* misc() const { return reinterpret_cast<uint32_t*>(base + a->misc_off); }
    __device__ uint32_t* maxbits() const { return reinterpret_cast<uint32_t*>(base + a->misc_off + 64); }
    __device__ float* sig_in() const { return reinterpret_cast<float*>(base + a->misc_off + 128); }
    __device__ float* sig_out() const { return reinterpret_cast<float*>(base + a->misc_off + 192); }
    __device__ float* z() const { return reinterpret_cast<float*>(base + a->z_off); }
    __device__ float* part() const { return reinterpret_cast<float*>(base + a->part_off); }
    __device__ uint8_t* b() const { return base + a->b_off; }
    __device__ uint8_t* stage(int s) const { return base + a->stage_off + static_cast<size_t>(s) * kStageBytes; }
};

// sigma per activation row, the B tiles and the per-block zero-point sums for the CTA's nblk
// blocks (decode warps only; ends with the B writes visible to the tensor core).
template <int TYPE, int MC>
__device__ void fill_operands(const Smem& sm, const float* xs, int nblk, int M) {
    using F = PnFmt<TYPE>;
    constexpr int STEPS = F::PAIRS;
    constexpr int PARTS = (MC == 16) ? 2 : 1;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int klen = nblk * F::BLK;
    uint32_t* maxbits = sm.maxbits();
    float* sig_in = sm.sig_in();
    float* sig_out = sm.sig_out();
    // sigma: max |x| over the slice per row m (the bit pattern of a non-negative float orders
    // like the value)
    const uint4* xv = reinterpret_cast<const uint4*>(xs);
    const int nvec = klen / 4;
    for (int m = 0; m < M; ++m) {
        uint32_t mx = 0;
        for (int i = tid; i < nvec; i += kDecodeThreads) {
            const uint4 v = xv[m * nvec + i];
            mx = max(mx, max(max(v.x & 0x7FFFFFFFu, v.y & 0x7FFFFFFFu), max(v.z & 0x7FFFFFFFu, v.w & 0x7FFFFFFFu)));
        }
        mx = __reduce_max_sync(0xffffffffu, mx);
        if (lane == 0) atomicMax(&maxbits[m], mx);
    }
    named_sync(1, kDecodeThreads);
    if (tid < M) {
        const uint32_t bits = maxbits[tid];
        const int E = static_cast<int>(bits >> 23);
        int sg = (bits == 0 || E >= 255) ? 0 : 141 - E;  // max < 2^(E-126)
        sg = min(100, max(-100, sg));
        sig_in[tid] = exp2i(sg);
        sig_out[tid] = exp2i(24 - sg);  // undoes sigma and the 2^-24 of the subnormal codes
    }
    named_sync(1, kDecodeThreads);
    // B tiles: one 16-byte chunk (8 k values of one column) per item; eight consecutive items
    // fill one 128-byte core matrix
    uint8_t* bbase = sm.b();
    const int tiles = nblk * STEPS * PARTS;
    for (int it = tid; it < tiles * 32; it += kDecodeThreads) {
        const int chunk = it & 31, tile = it >> 5;
        const int ng = chunk >> 4, kg = (chunk >> 3) & 1, n = ng * 8 + (chunk & 7);
        const int p = tile % PARTS, bj = tile / PARTS;
        const int j = bj % STEPS, blk = bj / STEPS;
        const int m = (MC == 16) ? n : (n >> 1);
        const int prt = (MC == 16) ? p : (n & 1);
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (m < M) {
            const float sc = sig_in[m] * step_scale<TYPE>(j);
            const float* xb = xs + m * klen + blk * F::BLK;
            const int odd = blk & 1;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int i = kg * 4 + q;  // decode register: k = 2i (low half), 2i + 1 (high half)
                const __half lo = split_part(xb[pn_elem(F::CPW, odd, i, j, 0)] * sc, prt);
                const __half hi = split_part(xb[pn_elem(F::CPW, odd, i, j, 1)] * sc, prt);
                w[q] = pack_half2(lo, hi);
            }
        }
        *reinterpret_cast<uint4*>(bbase + tile * kBTile + ng * kSbo + kg * kLbo + (chunk & 7) * 16) =
            make_uint4(w[0], w[1], w[2], w[3]);
    }
    // Z = z * sum over the block of (2^-24 * 8^j) * (hi + lo): one warp per (block, m)
    float* z = sm.z();
    for (int pr = warp; pr < nblk * M; pr += kDecodeWarps) {
        const int blk = pr / M, m = pr - blk * M;
        const float* xb = xs + m * klen + blk * F::BLK;
        const float si = sig_in[m];
        float s = 0.0f;
        for (int e = lane; e < F::BLK; e += 32) {
            const int j = (e % F::CPW) >> 1;
            const float v = xb[e] * (si * step_scale<TYPE>(j));
            const float hi = __half2float(__float2half_rn(v));
            const float lo = __half2float(__float2half_rn(v - hi));
            s = fmaf(5.9604644775390625e-08f * step_scale_inv<TYPE>(j), hi + lo, s);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) z[blk * M + m] = static_cast<float>(F::Z) * s;
    }
    fence_proxy_async_smem();
    named_sync(1, kDecodeThreads);
}

// Fold one block's D (read with tmem_ld) into the row sums: acc += d * (D - Z).
template <int MC, int NC>
__device__ __forceinline__ void fold_block(const uint32_t (&v)[NC], float d, const float* z, int M, float (&acc)[MC]) {
#pragma unroll
    for (int m = 0; m < MC; ++m) {
        if (m < M) {
            const float dv =
                (MC == 16) ? __uint_as_float(v[m]) : __uint_as_float(v[2 * m]) + __uint_as_float(v[2 * m + 1]);
            acc[m] = fmaf(d, dv - z[m], acc[m]);
        }
    }
}

template <int TYPE, int MC, int H>
__device__ void decode_loop(const Smem& sm, const TcArgs& a, uint32_t tbase, long long i0, int n_items, int u0) {
    using SHP = TcShape<TYPE>;
    constexpr int STEPS = PnFmt<TYPE>::PAIRS;
    constexpr int NC = (MC == 16) ? 16 : 2 * MC;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3;
    const int r = 32 * q + lane;
    const uint32_t set = tbase + (static_cast<uint32_t>(32 * q) << 16) + H * SHP::SETCOLS;
    const float* z = sm.z();
    const float* sig_out = sm.sig_out();
    float* part = sm.part();
    float acc[MC];
#pragma unroll
    for (int m = 0; m < MC; ++m) acc[m] = 0.0f;
    float dp[kSetBlocks] = {0.0f, 0.0f, 0.0f, 0.0f};
    int prev_lu = 0;
    bool ok = true;

    auto emit = [&](int j) {  // the rows of item j, scaled back, to the reducer
        const int buf = j & 1;
        if (j >= 2 && !mbar_wait_warp(sm.part_free(buf), ((j >> 1) - 1) & 1)) {
            ok = false;
            return;
        }
        float* dst = part + (H * 2 + buf) * a.M * kTileRows + r;
#pragma unroll
        for (int m = 0; m < MC; ++m) {
            if (m < a.M) dst[m * kTileRows] = acc[m] * sig_out[m];
            acc[m] = 0.0f;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.part_full(buf));
    };
    // Block slot BI: fold the previous item's D (when there is one), decode this item's block
    // into A, hand the slot to the MMA thread.
    auto block_step = [&](auto bi_c, int g, const uint32_t(&win)[36], bool decode) {
        constexpr int BI = decltype(bi_c)::value;
        const uint32_t a_col = set + BI * 8 * STEPS;
        const uint32_t d_col = set + SHP::ACOLS + kN * BI;
        uint32_t v[NC];
        if (g > 0) {
            if (!mbar_wait_warp(sm.slot_done(H, BI), (g - 1) & 1)) {
                ok = false;
                return;
            }
            tc_fence_after();
            tmem_ld<NC>(d_col, v);
        }
        float dn = 0.0f;
        if (decode) dn = decode_block<TYPE, H, BI>(win, a_col);
        if (g > 0) {
            tmem_wait_ld();
            fold_block<MC, NC>(v, dp[BI], z + (prev_lu * kUnitBlocks + kSetBlocks * H + BI) * a.M, a.M, acc);
        }
        dp[BI] = dn;
        if (decode) {
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.slot_full(H, BI));
        }
    };
    uint32_t win[36];
    for (int g = 0; g < n_items; ++g) {
        const long long i = i0 + g;
        const int lu = static_cast<int>(i / a.T) - u0;
        const int s = g % a.NS;
        if (!mbar_wait_warp(sm.full(s), (g / a.NS) & 1)) {
            ok = false;
            break;
        }
        const uint4* src = reinterpret_cast<const uint4*>(sm.stage(s) + r * kUnitBytes + 128 * H);
#pragma unroll
        for (int v = 0; v < 9; ++v) {
            const uint4 t = src[v];
            win[4 * v] = t.x;
            win[4 * v + 1] = t.y;
            win[4 * v + 2] = t.z;
            win[4 * v + 3] = t.w;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.empty(s));
        block_step(std::integral_constant<int, 0>{}, g, win, true);
        if (ok) block_step(std::integral_constant<int, 1>{}, g, win, true);
        if (ok) block_step(std::integral_constant<int, 2>{}, g, win, true);
        if (ok) block_step(std::integral_constant<int, 3>{}, g, win, true);
        if (!ok) break;
        if (g > 0) {
            emit(g - 1);
            if (!ok) break;
        }
        prev_lu = lu;
    }
    if (ok && n_items > 0) {
        // fold the last item's D blocks
        block_step(std::integral_constant<int, 0>{}, n_items, win, false);
        if (ok) block_step(std::integral_constant<int, 1>{}, n_items, win, false);
        if (ok) block_step(std::integral_constant<int, 2>{}, n_items, win, false);
        if (ok) block_step(std::integral_constant<int, 3>{}, n_items, win, false);
        if (ok) emit(n_items - 1);
    }
    if (!ok && lane == 0) record_error(a.err, kErrFullWait);
}

template <int TYPE, int MC>
__global__ void __launch_bounds__(kThreads, 1) pn_tc_gemv_kernel(const __grid_constant__ TcArgs a) {
    using F = PnFmt<TYPE>;
    using SHP = TcShape<TYPE>;
    constexpr int STEPS = F::PAIRS;
    constexpr int PARTS = (MC == 16) ? 2 : 1;
    constexpr int UK = kUnitBlocks * F::BLK;  // weights of a row per unit
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Smem sm{smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u), &a};
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // this CTA's share of the items, and the K units it touches
    const long long G = gridDim.x, c = blockIdx.x;
    const long long i0 = c * a.items / G, i1 = (c + 1) * a.items / G;
    const int n_items = static_cast<int>(i1 - i0);
    const int u0 = static_cast<int>(i0 / a.T);
    const int span = n_items > 0 ? static_cast<int>((i1 - 1) / a.T) - u0 + 1 : 0;
    const int nblk = span * kUnitBlocks;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.NS; ++s) {
            mbar_init(sm.full(s), 1);
            mbar_init(sm.empty(s), kDecodeWarps);
        }
        mbar_init(sm.x_ready(), 1);
        mbar_init(sm.x_free(), 1);
        for (int h = 0; h < 2; ++h) {
            for (int bi = 0; bi < kSetBlocks; ++bi) {
                mbar_init(sm.slot_full(h, bi), 4);
                mbar_init(sm.slot_done(h, bi), 1);
            }
            mbar_init(sm.part_full(h), kDecodeWarps);
            mbar_init(sm.part_free(h), 1);
        }
        mbar_fence_init();
        griddep_launch_dependents();
    }
    if (threadIdx.x < 16) sm.maxbits()[threadIdx.x] = 0u;
    if (warp == kMmaWarp) tmem_alloc(smem_addr(sm.misc()), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = sm.misc()[0];

    if (warp == kProducerWarp) {
        // ---------------- producer: x slice + one tensor-map copy per item ----------------
        if (lane == 0 && n_items > 0) {
            const uint64_t pol = l2_policy_evict_first();
            bool ok = true;
            auto issue = [&](int g) {
                const long long i = i0 + g;
                const int u = static_cast<int>(i / a.T);
                const int t = static_cast<int>(i - static_cast<long long>(u) * a.T);
                const int s = g % a.NS;
                if (g >= a.NS) {
                    if (!mbar_wait_bounded(sm.empty(s), ((g / a.NS) - 1) & 1)) return false;
                } else if (s >= a.x_stage) {
                    if (!mbar_wait_bounded(sm.x_free(), 0)) return false;
                }
                mbar_arrive_expect_tx(sm.full(s), static_cast<uint32_t>(kStageBytes));
                tma_load_2d(smem_addr(sm.stage(s)), &a.map, u * kUnitU32, t * kTileRows, sm.full(s), pol);
                return true;
            };
            int g = 0;
            if (a.flags & kStaticWeights) {
                // the weights are not written by earlier work in the stream: start streaming
                // them into the stages that will not hold x before the previous grid completes
                for (; ok && g < min(n_items, a.x_stage); ++g) ok = issue(g);
            }
            griddep_wait();
            // x rows: [m][nblk * BLK] fp32, one bulk copy per row (16-byte aligned: X is, and the
            // slice starts at a multiple of 512 elements)
            const uint32_t xbytes = static_cast<uint32_t>(nblk * F::BLK * 4);
            mbar_arrive_expect_tx(sm.x_ready(), xbytes * a.M);
            for (int m = 0; m < a.M; ++m)
                bulk_g2s_plain(smem_addr(sm.stage(a.x_stage)) + m * xbytes,
                               a.X + static_cast<size_t>(m) * a.K + static_cast<size_t>(u0) * UK, xbytes, sm.x_ready());
            for (; ok && g < n_items; ++g) ok = issue(g);
            if (!ok) record_error(a.err, kErrEmptyWait);
            // every copy issued has landed before the CTA may exit
            bool drained = mbar_wait_bounded(sm.x_ready(), 0);
            for (int gg = max(0, g - a.NS); drained && gg < g; ++gg)
                drained = mbar_wait_bounded(sm.full(gg % a.NS), (gg / a.NS) & 1);
            if (!drained) record_error(a.err, kErrDrainWait);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issue: one thread ----------------
        if (lane == 0 && n_items > 0) {
            const uint64_t desc0 = smem_desc_kmajor(smem_addr(sm.b()), kLbo, kSbo);
            int commits[2][kSetBlocks] = {};
            bool ok = true;
            for (int g = 0; g < n_items && ok; ++g) {
                const long long i = i0 + g;
                const int lu = static_cast<int>(i / a.T) - u0;
                for (int bi = 0; bi < kSetBlocks && ok; ++bi) {
                    for (int h = 0; h < 2; ++h) {
                        if (!mbar_wait_bounded(sm.slot_full(h, bi), g & 1)) {
                            record_error(a.err, kErrFullWait);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t set = tbase + h * SHP::SETCOLS;
                        const int blk = lu * kUnitBlocks + kSetBlocks * h + bi;
                        const uint32_t dcol = set + SHP::ACOLS + kN * bi;
#pragma unroll
                        for (int j = 0; j < STEPS; ++j)
#pragma unroll
                            for (int p = 0; p < PARTS; ++p) {
                                const uint32_t boff = static_cast<uint32_t>(((blk * STEPS + j) * PARTS + p) * kBTile);
                                tc_mma_f16_ts(dcol, set + bi * 8 * STEPS + 8 * j, desc0 + (boff >> 4), kIdesc,
                                              (j | p) != 0 ? 1u : 0u);
                            }
                        tc_commit(sm.slot_done(h, bi));
                        ++commits[h][bi];
                    }
                }
            }
            // every MMA issued has completed before tensor memory is released
            for (int h = 0; h < 2; ++h)
                for (int bi = 0; bi < kSetBlocks; ++bi)
                    if (commits[h][bi] > 0 && !mbar_wait_bounded(sm.slot_done(h, bi), (commits[h][bi] - 1) & 1))
                        record_error(a.err, kErrDrainWait);
        }
        __syncwarp();
    } else if (warp == kReducerWarp) {
        // ---------------- reducer: partial rows -> workspace -> Y ----------------
        if (n_items > 0) {
            griddep_wait();  // the workspace, the counters and Y belong to earlier grids until now
            const float* part = sm.part();
            bool ok = true;
            for (int j = 0; j < n_items; ++j) {
                const int buf = j & 1;
                if (!mbar_wait_warp(sm.part_full(buf), (j >> 1) & 1)) {
                    ok = false;
                    break;
                }
                const long long i = i0 + j;
                const int u = static_cast<int>(i / a.T);
                const int t = static_cast<int>(i - static_cast<long long>(u) * a.T);
                float* slot = a.ws + (static_cast<size_t>(t) * a.U + u) * a.M * kTileRows;
                for (int m = 0; m < a.M; ++m) {
                    const float4 p0 = reinterpret_cast<const float4*>(part + ((0 * 2 + buf) * a.M + m) * kTileRows)[lane];
                    const float4 p1 = reinterpret_cast<const float4*>(part + ((1 * 2 + buf) * a.M + m) * kTileRows)[lane];
                    __stcg(reinterpret_cast<float4*>(slot + m * kTileRows) + lane,
                           make_float4(p0.x + p1.x, p0.y + p1.y, p0.z + p1.z, p0.w + p1.w));
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(sm.part_free(buf));
                __threadfence();
                __syncwarp();
                unsigned old = 0;
                if (lane == 0) old = atomicAdd(a.cnt + t, 1u);
                old = __shfl_sync(0xffffffffu, old, 0);
                if (old == static_cast<unsigned>(a.U - 1)) {
                    // last item of row tile t: sum its U slots in unit order
                    __threadfence();
                    const int row = t * kTileRows + 4 * lane;
                    for (int m = 0; m < a.M; ++m) {
                        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                        for (int uu = 0; uu < a.U; ++uu) {
                            const float4 v = __ldcg(reinterpret_cast<const float4*>(
                                                        a.ws + ((static_cast<size_t>(t) * a.U + uu) * a.M + m) * kTileRows) +
                                                    lane);
                            acc.x += v.x;
                            acc.y += v.y;
                            acc.z += v.z;
                            acc.w += v.w;
                        }
                        float* y = a.Y + static_cast<size_t>(m) * a.N;
                        if (row + 0 < a.N) y[row + 0] = acc.x;
                        if (row + 1 < a.N) y[row + 1] = acc.y;
                        if (row + 2 < a.N) y[row + 2] = acc.z;
                        if (row + 3 < a.N) y[row + 3] = acc.w;
                    }
                    __syncwarp();
                    if (lane == 0) a.cnt[t] = 0u;  // ready for the next launch
                }
            }
            if (!ok && lane == 0) record_error(a.err, kErrReduceWait);
        }
    } else {
        // ---------------- decode warps ----------------
        if (n_items > 0) {
            if (named_sync_and(1, kDecodeThreads, mbar_wait_bounded(sm.x_ready(), 0))) {
                const float* xs = reinterpret_cast<const float*>(sm.stage(a.x_stage));
                fill_operands<TYPE, MC>(sm, xs, nblk, a.M);
                if (threadIdx.x == 0) mbar_arrive(sm.x_free());  // the x stages may now take weights
                if (warp < 4)
                    decode_loop<TYPE, MC, 0>(sm, a, tbase, i0, n_items, u0);
                else
                    decode_loop<TYPE, MC, 1>(sm, a, tbase, i0, n_items, u0);
            } else if (threadIdx.x == 0) {
                record_error(a.err, kErrFullWait);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
}

// ---- host side --------------------------------------------------------------------------------------

uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

struct Plan {
    int G = 0, NS = 0, x_stage = 0, span_max = 0;
    uint32_t bar_off = 0, misc_off = 0, z_off = 0, part_off = 0, b_off = 0, stage_off = 0, total = 0;
};

// Grid, stage count and shared-memory layout; false when the shape does not fit.
bool make_plan(int blk_weights, int steps, int parts, int M, int64_t T, int64_t U, int sms, Plan& p) {
    const int64_t items = T * U;
    p.G = static_cast<int>(std::min<int64_t>(sms, items));
    p.span_max = 0;
    for (int64_t c = 0; c < p.G; ++c) {
        const int64_t i0 = c * items / p.G, i1 = (c + 1) * items / p.G;
        if (i1 > i0) p.span_max = std::max<int>(p.span_max, static_cast<int>((i1 - 1) / T - i0 / T + 1));
    }
    const uint32_t nblk = static_cast<uint32_t>(p.span_max) * kUnitBlocks;
    p.bar_off = 0;
    p.misc_off = 8u * (2 * kMaxStages + 22);
    p.z_off = align_up(p.misc_off + 256u, 16);
    p.part_off = align_up(p.z_off + nblk * M * 4u, 16);
    p.b_off = align_up(p.part_off + 4u * M * kTileRows * 4u, 1024);
    p.stage_off = align_up(p.b_off + nblk * steps * parts * kBTile, 1024);
    const uint64_t xbytes = static_cast<uint64_t>(M) * nblk * blk_weights * 4u;
    const int x_stages = static_cast<int>((xbytes + kStageBytes - 1) / kStageBytes);
    for (int ns = kMaxStages; ns >= 2; --ns) {
        const uint64_t total = p.stage_off + static_cast<uint64_t>(ns) * kStageBytes;
        if (total + 1024u <= kSmemLimit && ns >= x_stages) {
            p.NS = ns;
            p.x_stage = ns - x_stages;
            p.total = static_cast<uint32_t>(total);
            return true;
        }
    }
    return false;
}

template <int TYPE, int MC>
cudaError_t launch_mc(TcArgs& a, bool static_weights, cudaStream_t stream) {
    using F = PnFmt<TYPE>;
    constexpr int PARTS = (MC == 16) ? 2 : 1;
    Plan p;
    if (!make_plan(F::BLK, F::PAIRS, PARTS, a.M, a.T, a.U, device_sm_count(), p)) return cudaErrorNotSupported;
    auto kern = pn_tc_gemv_kernel<TYPE, MC>;
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
    e = stream_workspace(stream, static_cast<size_t>(a.T) * a.U * a.M * kTileRows, static_cast<size_t>(a.T), &a.ws,
                         &a.cnt);
    if (e != cudaSuccess) return e;
    a.NS = p.NS;
    a.x_stage = p.x_stage;
    a.flags = static_weights ? kStaticWeights : 0u;
    a.bar_off = p.bar_off;
    a.misc_off = p.misc_off;
    a.z_off = p.z_off;
    a.part_off = p.part_off;
    a.b_off = p.b_off;
    a.stage_off = p.stage_off;
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(p.G, 1, 1);
    lc.blockDim = dim3(kThreads, 1, 1);
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
cudaError_t launch_typed(TcArgs& a, bool static_weights, cudaStream_t stream) {
    if (a.M <= 1) return launch_mc<TYPE, 1>(a, static_weights, stream);
    if (a.M <= 2) return launch_mc<TYPE, 2>(a, static_weights, stream);
    if (a.M <= 4) return launch_mc<TYPE, 4>(a, static_weights, stream);
    if (a.M <= 8) return launch_mc<TYPE, 8>(a, static_weights, stream);
    return launch_mc<TYPE, 16>(a, static_weights, stream);
}

}  // namespace

cudaError_t launch_pn_gemv_tc(int type, const uint8_t* W, int64_t N, int64_t K, const float* X, int M, float* Y,
                              int* err, bool static_weights, cudaStream_t stream) {
    if (N == 0) return cudaSuccess;
    const int blk = (type == kTypePn3t) ? 80 : 64;
    const int64_t nb = K / blk;
    if (nb % kUnitBlocks != 0 || M < 1 || M > 16) return cudaErrorNotSupported;
    const int64_t U = nb / kUnitBlocks, T = (N + kTileRows - 1) / kTileRows;
    if (N > INT32_MAX || K > INT32_MAX || U * kUnitU32 > INT32_MAX || T * kTileRows > INT32_MAX) return cudaErrorNotSupported;
    if (reinterpret_cast<uintptr_t>(W) % 16 != 0 || reinterpret_cast<uintptr_t>(X) % 16 != 0)
        return cudaErrorNotSupported;
    TcArgs a{};
    if (!encode_u32_map(&a.map, W, N, nb * kBlockBytes / 4, kUnitU32, kTileRows)) return cudaErrorNotSupported;
    a.X = X;
    a.Y = Y;
    a.err = err;
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.M = M;
    a.T = static_cast<int>(T);
    a.U = static_cast<int>(U);
    a.items = T * U;
    return (type == kTypePn3t) ? launch_typed<kTypePn3t>(a, static_weights, stream)
                               : launch_typed<kTypePn4t>(a, static_weights, stream);
}

}  // namespace pnq
