// pnq_gemv_mma.cu -- tensor-core GEMV straight from block-quantized weights (fast path).
//
// What it computes: Y[m][n] = sum_k w[n][k] x[m][k] for 1 <= M <= 16, w decoded in registers
// just before the multiply ("PN weight format", sections Block layout and Value; TandemLLM
// "Quantisation and profiles", section NVFP4: unpack 4-bit codes to 16-bit numbers in
// registers and multiply on the tensor cores).
//
// Structure of one CTA (RW consumer warps + 1 producer warp):
//  * The CTA owns R = 16*RW consecutive weight rows and one K slice; S CTAs of a cluster
//    split K and reduce their partial rows through distributed shared memory, in rank
//    order (deterministic, no atomics, no global scratch).
//  * The producer warp streams the slice HBM -> shared memory with 1-D bulk copies (one
//    per row per stage, 16-byte aligned: a chunk of 8 PN blocks is 272 = 17 x 16 bytes)
//    into an NS-stage ring guarded by mbarriers; the L2 policy is evict-first.
//  * Meanwhile the consumer warps turn the slice of x into mma B fragments in shared
//    memory: x is scaled by a power of two 2^sigma chosen per CTA from max|x| (so any
//    finite magnitude fits fp16) and split into fp16 hi + lo parts (about 22 bits),
//    one mma column each; M rows of x use 2M columns (NT = ceil(2M/8) n8 tiles).
//  * Each consumer warp decodes its 16 rows: a 32-bit word gives two codes at the same
//    shift in its two 16-bit halves, so one LOP3 builds an f16x2 of (1024 + n) and one
//    HADD2/HFMA2 makes it exactly n - z -- an mma A register with no conversion. Within a
//    block the k order is free (x is permuted the same way), which lets 2-byte aligned
//    words be read as aligned words that pair the high half of word i-1 with the low half
//    of word i. Each block's mma sum is scaled once by fp32(d) (PN); NVFP4 folds the
//    E4M3FN group scale into A with one HMUL2 (e2m1 * e4m3 is exact in fp16) and applies
//    the global multiplier at the end.
//  * Every mbarrier wait is bounded in time; a wait that gives up records a site code in
//    the library's device error word and the CTA skips its remaining work.
#include "pnq_device.cuh"
#include "pnq_internal.h"

#include <algorithm>
#include <cstdlib>
#include <cstring>

namespace pnq {
namespace {

constexpr int kMaxM = 16;

__host__ __device__ constexpr uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// Shared-memory map, computed identically on host and device.
struct Layout {
    uint32_t bar_off;      // full[NS], empty[NS], x-ready mbarriers
    uint32_t misc_off;     // maxbits[16] u32, sig_in[16] f32, sig_out[16] f32, issued u32
    uint32_t part_off;     // [R][M] f32 partial results (cluster reduction)
    uint32_t xs_off;       // the CTA's slice of x, [M][klen] as stored in global memory
    uint32_t bfrag_off;    // B fragments of the CTA's K slice
    uint32_t bfrag_unit;   // bytes of B fragments per block (PN) / 256-weight unit (NVFP4)
    uint32_t stage_off;    // NS stages
    uint32_t stage_bytes;  // bytes per stage
    uint32_t pitch;        // bytes per row in a stage (codes for NVFP4)
    uint32_t pitch_s;      // NVFP4: bytes per row of the stage's scale area
    uint32_t scale_off;    // NVFP4: offset of the scale area inside a stage
    uint32_t total;
};

// Stage pitch: a multiple of 16 bytes whose quotient by 16 is odd, so the 8 row groups of
// a warp fall on distinct 16-byte bank groups.
__host__ __device__ constexpr uint32_t odd16_pitch(uint32_t bytes) {
    return ((align_up(bytes, 16) / 16) % 2 == 1) ? align_up(bytes, 16) : align_up(bytes, 16) + 16;
}

// unit_k: weights per unit (BLK for PN, 256 for NVFP4); x_bytes: bytes per x element.
__host__ __device__ inline Layout make_layout(bool nvfp4, int steps_per_unit, int M, int units_max, int unit_k,
                                              int x_bytes, int R, int chunk, int NS) {
    Layout L{};
    L.bar_off = 0;
    L.misc_off = align_up(8u * (2 * NS + 1), 16);
    L.part_off = L.misc_off + 256;
    L.xs_off = align_up(L.part_off + 4u * R * M, 128);
    L.bfrag_off = align_up(L.xs_off + static_cast<uint32_t>(M) * units_max * unit_k * x_bytes, 128);
    L.bfrag_unit = 64u * M * steps_per_unit;  // 8M lanes x steps x 8 bytes
    L.stage_off = align_up(L.bfrag_off + L.bfrag_unit * units_max, 128);
    if (!nvfp4) {
        L.pitch = odd16_pitch(34u * chunk);
        L.pitch_s = 0;
        L.scale_off = 0;
        L.stage_bytes = align_up(L.pitch * R, 128);
    } else {
        L.pitch = odd16_pitch(128u * chunk);
        L.pitch_s = odd16_pitch(16u * chunk);
        L.scale_off = align_up(L.pitch * R, 128);
        L.stage_bytes = align_up(L.scale_off + L.pitch_s * R, 128);
    }
    L.total = L.stage_off + L.stage_bytes * NS;
    return L;
}

struct Args {
    const uint8_t* W;       // PN blocks, or NVFP4 codes
    const uint8_t* scales;  // NVFP4 scales
    const void* X;          // fp32 (PN) or bf16 (NVFP4), [M][K]
    float* Y;               // [M][N]
    int* err;
    float g;                // NVFP4 global multiplier
    int N;
    int K;
    int units;              // blocks per row (PN) or 256-weight units per row (NVFP4)
    int M;
    int S;                  // cluster size along K
    int NS;                 // stages
    int chunk;              // units per stage
};

// ---- per-CTA setup shared by both formats ----------------------------------------------

struct Slice {
    int u0;       // first unit of this CTA's slice
    int nunits;   // units in the slice
    int nchunks;
};

__device__ __forceinline__ Slice cta_slice(const Args& a, uint32_t rank, int align_units) {
    // Split units into S slices, each a multiple of align_units (8 blocks for PN so that a
    // chunk row is a whole number of 16-byte lines).
    const int U = a.units / align_units;
    const int g0 = static_cast<int>((static_cast<int64_t>(rank) * U) / a.S);
    const int g1 = static_cast<int>((static_cast<int64_t>(rank + 1) * U) / a.S);
    Slice s;
    s.u0 = g0 * align_units;
    s.nunits = (g1 - g0) * align_units;
    s.nchunks = (s.nunits + a.chunk - 1) / a.chunk;
    return s;
}

// x element k of row m of the CTA's slice, from the shared-memory copy (fp32 or bf16).
template <bool BF16_X>
__device__ __forceinline__ float xs_at(const uint8_t* xs, int klen, int m, int k) {
    if (BF16_X)
        return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(xs)[m * klen + k]) << 16);
    return reinterpret_cast<const float*>(xs)[m * klen + k];
}

// Per-m power-of-two scaling: sigma chosen so max|x| * 2^sigma lies in [2^14, 2^15) over the
// CTA's slice (any finite x then fits fp16; an all-zero or non-finite slice keeps sigma = 0).
template <bool BF16_X>
__device__ void compute_sigma(const Args& a, int klen, uint8_t* smem, const Layout& L, int nct) {
    uint32_t* maxbits = reinterpret_cast<uint32_t*>(smem + L.misc_off);
    float* sig_in = reinterpret_cast<float*>(smem + L.misc_off + 64);
    float* sig_out = reinterpret_cast<float*>(smem + L.misc_off + 128);
    const int tid = threadIdx.x;
    const uint4* xv = reinterpret_cast<const uint4*>(smem + L.xs_off);
    const int per_vec = BF16_X ? 8 : 4;
    const int nvec = klen / per_vec;  // klen is a multiple of 64
    for (int m = 0; m < a.M; ++m) {
        uint32_t mx = 0;
        for (int i = tid; i < nvec; i += nct) {
            const uint4 v = xv[m * nvec + i];
            if (BF16_X) {
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) mx = max(mx, max((w[q] << 16) & 0x7FFFFFFFu, w[q] & 0x7FFF0000u));
            } else {
                mx = max(mx, max(max(v.x & 0x7FFFFFFFu, v.y & 0x7FFFFFFFu), max(v.z & 0x7FFFFFFFu, v.w & 0x7FFFFFFFu)));
            }
        }
        mx = __reduce_max_sync(0xffffffffu, mx);
        if ((tid & 31) == 0) atomicMax(&maxbits[m], mx);
    }
    named_sync(1, nct);
    if (tid < a.M) {
        const uint32_t bits = maxbits[tid];
        const int E = static_cast<int>(bits >> 23);
        int sg = (bits == 0 || E >= 255) ? 0 : 141 - E;  // max < 2^(E-126)
        sg = min(126, max(-126, sg));
        sig_in[tid] = exp2i(sg);
        sig_out[tid] = exp2i(-sg);
    }
    named_sync(1, nct);
}

// fp16 hi / lo parts of x * 2^sigma.
__device__ __forceinline__ __half split_part(float xs, int part) {
    const __half hi = __float2half_rn(xs);
    if (part == 0) return hi;
    return __float2half_rn(xs - __half2float(hi));
}

// B fragment store address for (unit, tile t, lane l, step st, register r).
__device__ __forceinline__ uint32_t bfrag_offset(const Layout& L, int M, int steps, int unit, int t, int l, int st,
                                                 int r) {
    const int LU = min(32, 8 * M - 32 * t);
    const int q = st >> 1;
    uint32_t off = L.bfrag_off + unit * L.bfrag_unit + t * (256 * steps);
    if ((steps & 1) && st == steps - 1)
        off += (steps >> 1) * LU * 16 + l * 8 + r * 4;
    else
        off += q * LU * 16 + l * 16 + (st & 1) * 8 + r * 4;
    return off;
}

// Loads this lane's B registers of one unit for tile t (zero where the column is unused).
template <int STEPS>
__device__ __forceinline__ void load_bfrag(const uint8_t* smem, const Layout& L, int M, int unit, int t, int lane,
                                           uint32_t (&b)[STEPS][2]) {
    const int LU = min(32, 8 * M - 32 * t);
    if (lane < LU) {
        const uint8_t* base = smem + L.bfrag_off + unit * L.bfrag_unit + t * (256 * STEPS);
#pragma unroll
        for (int q = 0; q < STEPS / 2; ++q) {
            const uint4 v = *reinterpret_cast<const uint4*>(base + q * LU * 16 + lane * 16);
            b[2 * q][0] = v.x;
            b[2 * q][1] = v.y;
            b[2 * q + 1][0] = v.z;
            b[2 * q + 1][1] = v.w;
        }
        if (STEPS & 1) {
            const uint2 v = *reinterpret_cast<const uint2*>(base + (STEPS / 2) * LU * 16 + lane * 8);
            b[STEPS - 1][0] = v.x;
            b[STEPS - 1][1] = v.y;
        }
    } else {
#pragma unroll
        for (int s = 0; s < STEPS; ++s) b[s][0] = b[s][1] = 0u;
    }
}

// ---- PN decode ------------------------------------------------------------------------

// Pair j of a (possibly re-paired) word: both halves hold a code at bits BITS*j; result is
// the f16x2 (n_lo - z, n_hi - z), exact.
template <int TYPE, int J>
__device__ __forceinline__ uint32_t pn_pair(uint32_t w) {
    constexpr uint32_t kMagic = 0x64006400u;  // 1024.0 in both halves
    if (TYPE == kTypePn3t) {
        // codes at bits 0-2, 3-5, 6-8 in place; bits 9-11 and 12-14 after a shift by 9
        constexpr int jj = (J < 3) ? J : J - 3;
        const uint32_t src = (J < 3) ? w : (w >> 9);
        const uint32_t mask = 0x00070007u << (3 * jj);
        const uint32_t h = lop3_and_or(src, mask, kMagic);  // 1024 + n * 8^jj
        if (jj == 0) return hadd2_u32(h, 0xE404E404u);                  // - 1028
        if (jj == 1) return hfma2_u32(h, 0x30003000u, 0xD820D820u);     // /8 - 132
        return hfma2_u32(h, 0x24002400u, 0xCD00CD00u);                  // /64 - 20
    } else {
        constexpr int jj = J & 1;
        const uint32_t src = (J < 2) ? w : (w >> 8);
        const uint32_t mask = 0x000F000Fu << (4 * jj);
        const uint32_t h = lop3_and_or(src, mask, kMagic);  // 1024 + n * 16^jj
        if (jj == 0) return hadd2_u32(h, 0xE408E408u);                  // - 1032
        return hfma2_u32(h, 0x2C002C00u, 0xD480D480u);                  // /16 - 72
    }
}

// Element index (within a block) of the low (hi_half = 0) or high code of pair j of decode
// word i, for a block starting on a 4-byte boundary (even block) or not (odd block).
// Odd block: natural word i (low half = even t = 2j, high half = odd t = 2j + 1).
// Even block: the aligned word at byte 4i holds the high half of word i-1 and the low half
// of word i; decode word 0 is built from the low half of word 0 and the high half of word 7.
__device__ __forceinline__ int pn_elem(int cpw, int odd_block, int i, int j, int hi_half) {
    if (odd_block) return cpw * i + 2 * j + hi_half;
    if (i == 0) return hi_half ? cpw * 7 + 2 * j + 1 : 2 * j;
    return hi_half ? cpw * i + 2 * j : cpw * (i - 1) + 2 * j + 1;
}

template <int TYPE, int NT>
__device__ void pn_fill_bfrag(const Args& a, const Slice& sl, uint8_t* smem, const Layout& L, int nct) {
    using F = PnFmt<TYPE>;
    constexpr int STEPS = F::PAIRS;
    const float* sig_in = reinterpret_cast<const float*>(smem + L.misc_off + 64);
    const uint8_t* xs = smem + L.xs_off;
    const int klen = sl.nunits * F::BLK;
    const int lanes = 8 * a.M;
    const int total = sl.nunits * lanes;
    for (int idx = threadIdx.x; idx < total; idx += nct) {
        const int u = idx / lanes;
        const int lr = idx - u * lanes;
        const int t = lr >> 5, l = lr & 31;
        const int g = l >> 2, tig = l & 3;
        const int col = 8 * t + g, m = col >> 1, part = col & 1;
        const int odd = u & 1;  // slices start on a multiple of 8 blocks
        const int kb = u * F::BLK;
        const float si = sig_in[m];
#pragma unroll
        for (int st = 0; st < STEPS; ++st) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int i = tig + 4 * r;
                const int e0 = pn_elem(F::CPW, odd, i, st, 0), e1 = pn_elem(F::CPW, odd, i, st, 1);
                const __half v0 = split_part(xs_at<false>(xs, klen, m, kb + e0) * si, part);
                const __half v1 = split_part(xs_at<false>(xs, klen, m, kb + e1) * si, part);
                *reinterpret_cast<uint32_t*>(smem + bfrag_offset(L, a.M, STEPS, u, t, l, st, r)) = pack_half2(v0, v1);
            }
        }
    }
}

template <int TYPE, int NT, int ODD>
__device__ __forceinline__ void pn_block(const uint8_t* r0p, const uint8_t* r1p, int bl, const uint8_t* smem,
                                         const Layout& L, int M, int unit, int lane, float (&acc)[NT][4]) {
    using F = PnFmt<TYPE>;
    constexpr int STEPS = F::PAIRS;
    const int tig = lane & 3;
    const int off = kBlockBytes * bl;
    const float d0 = __half2float(*reinterpret_cast<const __half*>(r0p + off));
    const float d1 = __half2float(*reinterpret_cast<const __half*>(r1p + off));
    uint32_t w0a, w0b, w1a, w1b;
    if (ODD) {
        w0a = *reinterpret_cast<const uint32_t*>(r0p + off + 2 + 4 * tig);
        w0b = *reinterpret_cast<const uint32_t*>(r0p + off + 18 + 4 * tig);
        w1a = *reinterpret_cast<const uint32_t*>(r1p + off + 2 + 4 * tig);
        w1b = *reinterpret_cast<const uint32_t*>(r1p + off + 18 + 4 * tig);
    } else {
        w0a = *reinterpret_cast<const uint32_t*>(r0p + off + 4 * tig);
        w0b = *reinterpret_cast<const uint32_t*>(r0p + off + 16 + 4 * tig);
        w1a = *reinterpret_cast<const uint32_t*>(r1p + off + 4 * tig);
        w1b = *reinterpret_cast<const uint32_t*>(r1p + off + 16 + 4 * tig);
        const uint32_t x0 = *reinterpret_cast<const uint32_t*>(r0p + off + 32);
        const uint32_t x1 = *reinterpret_cast<const uint32_t*>(r1p + off + 32);
        const uint32_t p0 = prmt(w0a, x0, 0x5432u), p1 = prmt(w1a, x1, 0x5432u);
        w0a = (tig == 0) ? p0 : w0a;
        w1a = (tig == 0) ? p1 : w1a;
    }
    float c[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) c[t][0] = c[t][1] = c[t][2] = c[t][3] = 0.0f;
    uint32_t b[NT][STEPS][2];
#pragma unroll
    for (int t = 0; t < NT; ++t) load_bfrag<STEPS>(smem, L, M, unit, t, lane, b[t]);
#define PNQ_STEP(J)                                                                                        \
    {                                                                                                      \
        const uint32_t a0 = pn_pair<TYPE, J>(w0a), a1 = pn_pair<TYPE, J>(w1a);                             \
        const uint32_t a2 = pn_pair<TYPE, J>(w0b), a3 = pn_pair<TYPE, J>(w1b);                             \
        _Pragma("unroll") for (int t = 0; t < NT; ++t) mma_f16_16816(c[t], a0, a1, a2, a3, b[t][J][0], b[t][J][1]); \
    }
    PNQ_STEP(0)
    PNQ_STEP(1)
    PNQ_STEP(2)
    PNQ_STEP(3)
    if constexpr (STEPS == 5) PNQ_STEP(4)
#undef PNQ_STEP
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        acc[t][0] = fmaf(d0, c[t][0], acc[t][0]);
        acc[t][1] = fmaf(d0, c[t][1], acc[t][1]);
        acc[t][2] = fmaf(d1, c[t][2], acc[t][2]);
        acc[t][3] = fmaf(d1, c[t][3], acc[t][3]);
    }
}

// ---- NVFP4 decode --------------------------------------------------------------------------
// A 256-weight unit of one row is 32 code words (8 codes each, one 16-weight group per two
// words) and 16 scale bytes. Lane tig owns words tig + 4q (q = 0..7). Step (q2, i) uses byte
// i of words tig + 8 q2 (A registers 0, 1) and tig + 8 q2 + 4 (registers 2, 3); a byte is
// the pair (k, k + 1) with k = 8 * word + 2 i.
constexpr int kNvSteps = 16;

__device__ __forceinline__ int nv_elem(int tig, int st, int r, int hi) {
    const int q2 = st >> 2, i = st & 3;
    return 8 * (tig + 8 * q2 + 4 * r) + 2 * i + hi;
}

template <int NT>
__device__ void nv_fill_bfrag(const Args& a, const Slice& sl, uint8_t* smem, const Layout& L, int nct) {
    const float* sig_in = reinterpret_cast<const float*>(smem + L.misc_off + 64);
    const uint8_t* xs = smem + L.xs_off;
    const int klen = sl.nunits * 256;
    const int lanes = 8 * a.M;
    const int total = sl.nunits * lanes;
    for (int idx = threadIdx.x; idx < total; idx += nct) {
        const int u = idx / lanes;
        const int lr = idx - u * lanes;
        const int t = lr >> 5, l = lr & 31;
        const int g = l >> 2, tig = l & 3;
        const int col = 8 * t + g, m = col >> 1, part = col & 1;
        const int kb = u * 256;
        const float si = sig_in[m];
#pragma unroll 4
        for (int st = 0; st < kNvSteps; ++st) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const __half v0 = split_part(xs_at<true>(xs, klen, m, kb + nv_elem(tig, st, r, 0)) * si, part);
                const __half v1 = split_part(xs_at<true>(xs, klen, m, kb + nv_elem(tig, st, r, 1)) * si, part);
                *reinterpret_cast<uint32_t*>(smem + bfrag_offset(L, a.M, kNvSteps, u, t, l, st, r)) = pack_half2(v0, v1);
            }
        }
    }
}

template <int NT>
__device__ __forceinline__ void nv_unit(const uint8_t* c0p, const uint8_t* c1p, const uint8_t* s0p,
                                        const uint8_t* s1p, const uint8_t* smem, const Layout& L, int M, int unit,
                                        int lane, float (&acc)[NT][4]) {
    const int tig = lane & 3;
    const uint32_t ssel = (tig >> 1) | (((tig >> 1) + 2) << 4);  // bytes tig/2 and tig/2 + 2
#pragma unroll
    for (int q2 = 0; q2 < 4; ++q2) {
        const uint32_t w0a = *reinterpret_cast<const uint32_t*>(c0p + 4 * (tig + 8 * q2));
        const uint32_t w0b = *reinterpret_cast<const uint32_t*>(c0p + 4 * (tig + 8 * q2 + 4));
        const uint32_t w1a = *reinterpret_cast<const uint32_t*>(c1p + 4 * (tig + 8 * q2));
        const uint32_t w1b = *reinterpret_cast<const uint32_t*>(c1p + 4 * (tig + 8 * q2 + 4));
        // scales of groups 4 q2 + tig/2 (words tig + 8 q2) and 4 q2 + 2 + tig/2 (+4)
        const uint32_t sc0 = e4m3x2_to_f16x2(prmt(*reinterpret_cast<const uint32_t*>(s0p + 4 * q2), 0u, ssel));
        const uint32_t sc1 = e4m3x2_to_f16x2(prmt(*reinterpret_cast<const uint32_t*>(s1p + 4 * q2), 0u, ssel));
        const uint32_t s0a = prmt(sc0, sc0, 0x1010u), s0b = prmt(sc0, sc0, 0x3232u);
        const uint32_t s1a = prmt(sc1, sc1, 0x1010u), s1b = prmt(sc1, sc1, 0x3232u);
        uint32_t b[NT][4][2];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int LU = min(32, 8 * M - 32 * t);
            if (lane < LU) {
                const uint8_t* base = smem + L.bfrag_off + unit * L.bfrag_unit + t * (256 * kNvSteps);
                const uint4 v0 = *reinterpret_cast<const uint4*>(base + (2 * q2) * LU * 16 + lane * 16);
                const uint4 v1 = *reinterpret_cast<const uint4*>(base + (2 * q2 + 1) * LU * 16 + lane * 16);
                b[t][0][0] = v0.x; b[t][0][1] = v0.y; b[t][1][0] = v0.z; b[t][1][1] = v0.w;
                b[t][2][0] = v1.x; b[t][2][1] = v1.y; b[t][3][0] = v1.z; b[t][3][1] = v1.w;
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) b[t][i][0] = b[t][i][1] = 0u;
            }
        }
#define PNQ_NVSTEP(I)                                                                                    \
    {                                                                                                    \
        const uint32_t a0 = hmul2_u32(e2m1x2_to_f16x2<I>(w0a), s0a);                                     \
        const uint32_t a1 = hmul2_u32(e2m1x2_to_f16x2<I>(w1a), s1a);                                     \
        const uint32_t a2 = hmul2_u32(e2m1x2_to_f16x2<I>(w0b), s0b);                                     \
        const uint32_t a3 = hmul2_u32(e2m1x2_to_f16x2<I>(w1b), s1b);                                     \
        _Pragma("unroll") for (int t = 0; t < NT; ++t) mma_f16_16816(acc[t], a0, a1, a2, a3, b[t][I][0], b[t][I][1]); \
    }
        PNQ_NVSTEP(0)
        PNQ_NVSTEP(1)
        PNQ_NVSTEP(2)
        PNQ_NVSTEP(3)
#undef PNQ_NVSTEP
    }
}

// ---- the kernel ---------------------------------------------------------------------------------

template <int TYPE, int NT, int RW>
__global__ void __launch_bounds__(32 * (RW + 1)) gemv_mma_kernel(const Args a) {
    constexpr bool kNv = (TYPE == kTypeNvfp4);
    constexpr int R = 16 * RW;
    constexpr int kSteps = kNv ? kNvSteps : PnFmt<(kNv ? kTypePn4t : TYPE)>::PAIRS;
    constexpr int kAlignUnits = kNv ? 1 : 8;
    extern __shared__ __align__(128) uint8_t smem[];

    const uint32_t rank = (a.S > 1) ? cluster_ctarank() : 0u;
    const int units_max = kAlignUnits * ((a.units / kAlignUnits + a.S - 1) / a.S);
    constexpr int kUnitK = kNv ? 256 : PnFmt<(kNv ? kTypePn4t : TYPE)>::BLK;
    constexpr int kXBytes = kNv ? 2 : 4;
    const Layout L = make_layout(kNv, kSteps, a.M, units_max, kUnitK, kXBytes, R, a.chunk, a.NS);
    const Slice sl = cta_slice(a, rank, kAlignUnits);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = blockIdx.y * R;
    const int rows_valid = min(R, a.N - row0);
    const uint32_t bar0 = smem_addr(smem + L.bar_off);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (a.NS + s); };
    const uint32_t x_bar = bar0 + 8u * (2 * a.NS);
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L.misc_off);

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.NS; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), RW);
        }
        mbar_init(x_bar, 1);
        mbar_fence_init();
    }
    if (threadIdx.x < 16) misc[threadIdx.x] = 0u;  // maxbits
    if (threadIdx.x == 16) misc[48] = 0u;          // issued
    __syncthreads();

    if (warp == RW) {
        // ---------------- producer warp ----------------
        const uint64_t pol = l2_policy_evict_first();
        {
            // the CTA's slice of x: one bulk copy per activation row (16-byte aligned: X is,
            // and the slice starts at a multiple of 64 elements)
            const uint32_t xbytes = static_cast<uint32_t>(sl.nunits * kUnitK * kXBytes);
            if (lane == 0) mbar_arrive_expect_tx(x_bar, xbytes * a.M);
            __syncwarp();
            const uint8_t* xsrc = static_cast<const uint8_t*>(a.X) + static_cast<size_t>(sl.u0) * kUnitK * kXBytes;
            if (lane < a.M)
                bulk_g2s_plain(smem_addr(smem + L.xs_off) + lane * xbytes,
                               xsrc + static_cast<size_t>(lane) * a.K * kXBytes, xbytes, x_bar);
        }
        int issued = 0;
        if (!kNv) {
            const size_t rowbytes = static_cast<size_t>(a.units) * kBlockBytes;
            const uint8_t* src0 = a.W + static_cast<size_t>(row0) * rowbytes + static_cast<size_t>(sl.u0) * kBlockBytes;
            for (int c = 0; c < sl.nchunks; ++c) {
                const int s = c % a.NS;
                if (c >= a.NS && !mbar_wait_bounded(empty_bar(s), ((c / a.NS) - 1) & 1)) {
                    if (lane == 0) record_error(a.err, kErrEmptyWait);
                    break;
                }
                const uint32_t bytes = static_cast<uint32_t>(min(a.chunk, sl.nunits - c * a.chunk) * kBlockBytes);
                if (lane == 0) mbar_arrive_expect_tx(full_bar(s), bytes * rows_valid);
                __syncwarp();
                const uint32_t dst = smem_addr(smem + L.stage_off + s * L.stage_bytes);
                for (int r = lane; r < rows_valid; r += 32)
                    bulk_g2s(dst + r * L.pitch, src0 + r * rowbytes + static_cast<size_t>(c) * a.chunk * kBlockBytes,
                             bytes, full_bar(s), pol);
                issued = c + 1;
            }
        } else {
            const size_t rowc = static_cast<size_t>(a.K) / 2, rows_ = static_cast<size_t>(a.K) / 16;
            const uint8_t* c0 = a.W + static_cast<size_t>(row0) * rowc + static_cast<size_t>(sl.u0) * 128;
            const uint8_t* s0 = a.scales + static_cast<size_t>(row0) * rows_ + static_cast<size_t>(sl.u0) * 16;
            for (int c = 0; c < sl.nchunks; ++c) {
                const int s = c % a.NS;
                if (c >= a.NS && !mbar_wait_bounded(empty_bar(s), ((c / a.NS) - 1) & 1)) {
                    if (lane == 0) record_error(a.err, kErrEmptyWait);
                    break;
                }
                const int cu = min(a.chunk, sl.nunits - c * a.chunk);
                const uint32_t cbytes = 128u * cu, sbytes = 16u * cu;
                if (lane == 0) mbar_arrive_expect_tx(full_bar(s), (cbytes + sbytes) * rows_valid);
                __syncwarp();
                const uint32_t dst = smem_addr(smem + L.stage_off + s * L.stage_bytes);
                for (int r = lane; r < rows_valid; r += 32) {
                    bulk_g2s(dst + r * L.pitch, c0 + r * rowc + static_cast<size_t>(c) * a.chunk * 128, cbytes,
                             full_bar(s), pol);
                    bulk_g2s(dst + L.scale_off + r * L.pitch_s, s0 + r * rows_ + static_cast<size_t>(c) * a.chunk * 16,
                             sbytes, full_bar(s), pol);
                }
                issued = c + 1;
            }
        }
        if (lane == 0) misc[48] = static_cast<uint32_t>(issued);
    } else {
        // ---------------- consumer warps ----------------
        const int nct = 32 * RW;
        const int klen = sl.nunits * kUnitK;
        if (!mbar_wait_bounded(x_bar, 0) && lane == 0) record_error(a.err, kErrFullWait);
        compute_sigma<kNv>(a, klen, smem, L, nct);
        if constexpr (kNv)
            nv_fill_bfrag<NT>(a, sl, smem, L, nct);
        else
            pn_fill_bfrag<TYPE, NT>(a, sl, smem, L, nct);
        named_sync(1, nct);

        float acc[NT][4];
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;
        const int g = lane >> 2, tig = lane & 3;
        for (int c = 0; c < sl.nchunks; ++c) {
            const int s = c % a.NS;
            if (!mbar_wait_bounded(full_bar(s), (c / a.NS) & 1)) {
                if (lane == 0) record_error(a.err, kErrFullWait);
                break;
            }
            const uint8_t* st = smem + L.stage_off + s * L.stage_bytes;
            const int n_in = min(a.chunk, sl.nunits - c * a.chunk);
            if constexpr (!kNv) {
                const uint8_t* r0p = st + (16 * warp + g) * L.pitch;
                const uint8_t* r1p = r0p + 8 * L.pitch;
                for (int bl = 0; bl < n_in; bl += 2) {
                    pn_block<TYPE, NT, 0>(r0p, r1p, bl, smem, L, a.M, c * a.chunk + bl, lane, acc);
                    pn_block<TYPE, NT, 1>(r0p, r1p, bl + 1, smem, L, a.M, c * a.chunk + bl + 1, lane, acc);
                }
            } else {
                const uint8_t* c0p = st + (16 * warp + g) * L.pitch;
                const uint8_t* c1p = c0p + 8 * L.pitch;
                const uint8_t* s0p = st + L.scale_off + (16 * warp + g) * L.pitch_s;
                const uint8_t* s1p = s0p + 8 * L.pitch_s;
                for (int u = 0; u < n_in; ++u)
                    nv_unit<NT>(c0p + 128 * u, c1p + 128 * u, s0p + 16 * u, s1p + 16 * u, smem, L, a.M,
                                c * a.chunk + u, lane, acc);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar(s));
        }

        // epilogue: combine hi + lo columns, undo the power-of-two scaling
        const float* sig_out = reinterpret_cast<const float*>(smem + L.misc_off + 128);
        float* part = reinterpret_cast<float*>(smem + L.part_off);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int m = 4 * t + tig;
            if (m < a.M) {
                const float so = kNv ? sig_out[m] * a.g : sig_out[m];
                const float y0 = (acc[t][0] + acc[t][1]) * so;
                const float y1 = (acc[t][2] + acc[t][3]) * so;
                const int ra = 16 * warp + g, rb = ra + 8;
                if (a.S == 1) {
                    if (ra < rows_valid) a.Y[static_cast<size_t>(m) * a.N + row0 + ra] = y0;
                    if (rb < rows_valid) a.Y[static_cast<size_t>(m) * a.N + row0 + rb] = y1;
                } else {
                    part[ra * a.M + m] = y0;
                    part[rb * a.M + m] = y1;
                }
            }
        }
    }

    __syncthreads();
    // Drain: no CTA leaves while a bulk copy it issued may still be writing its shared memory.
    if (warp == RW && lane == 0) {
        if (!mbar_wait_bounded(x_bar, 0)) record_error(a.err, kErrDrainWait);
        const int issued = static_cast<int>(misc[48]);
        for (int c = max(0, issued - a.NS); c < issued; ++c)
            if (!mbar_wait_bounded(full_bar(c % a.NS), (c / a.NS) & 1)) record_error(a.err, kErrDrainWait);
    }
    if (a.S > 1) {
        cluster_sync();
        // rank r reduces rows r, r + S, ... over all ranks, in rank order
        const uint32_t part_addr = smem_addr(smem + L.part_off);
        for (int idx = threadIdx.x; idx < R * a.M; idx += blockDim.x) {
            const int r = idx / a.M, m = idx - r * a.M;
            if ((r % a.S) != static_cast<int>(rank) || r >= rows_valid) continue;
            float sum = 0.0f;
            for (int q = 0; q < a.S; ++q) sum += ld_dsmem_f32(part_addr + 4u * idx, static_cast<uint32_t>(q));
            a.Y[static_cast<size_t>(m) * a.N + row0 + r] = sum;
        }
        cluster_sync();
    }
}

// ---- host side --------------------------------------------------------------------------------------

template <int TYPE, int NT, int RW>
cudaError_t launch_one(const Args& a, int G, size_t smem_bytes, cudaStream_t stream) {
    auto kern = gemv_mma_kernel<TYPE, NT, RW>;
    // The shared-memory opt-in is raised once per device and size (not on every launch, and
    // so never while a stream is being captured after the first eager call).
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
    static bool wide[64] = {};
    if (a.S > 8 && !wide[dev]) {  // clusters of 9..16 CTAs are a non-portable opt-in
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        wide[dev] = true;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(a.S, G, 1);
    cfg.blockDim = dim3(32 * (RW + 1), 1, 1);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    cfg.numAttrs = 0;
    if (a.S > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = a.S;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int TYPE, int RW>
cudaError_t launch_nt(const Args& a, int G, size_t smem_bytes, cudaStream_t stream) {
    const int nt = (2 * a.M + 7) / 8;
    if (nt <= 1) return launch_one<TYPE, 1, RW>(a, G, smem_bytes, stream);
    if (nt <= 2) return launch_one<TYPE, 2, RW>(a, G, smem_bytes, stream);
    return launch_one<TYPE, 4, RW>(a, G, smem_bytes, stream);
}

// Environment override "rw,S,chunk,ns" (any field 0 = automatic), read once; used by the
// tile sweeps in the benchmark tooling.
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

cudaError_t launch_common(int type, Args a, int64_t N, MmaConfig cfg, cudaStream_t stream) {
    const bool nv = (type == kTypeNvfp4);
    const MmaConfig env = env_config();
    if (cfg.rw <= 0) cfg.rw = env.rw;
    if (cfg.S <= 0) cfg.S = env.S;
    if (cfg.cb <= 0) cfg.cb = env.cb;
    if (cfg.ns <= 0) cfg.ns = env.ns;
    const bool rw_forced = cfg.rw > 0, ns_forced = cfg.ns > 0, s_forced = cfg.S > 0;
    const int align_units = nv ? 1 : 8;
    const int U = a.units / align_units;
    if (U < 1 || N > INT32_MAX) return cudaErrorNotSupported;
    if (reinterpret_cast<uintptr_t>(a.X) % 16 != 0) return cudaErrorNotSupported;  // x slices are bulk-copied
    const int steps = nv ? kNvSteps : (type == kTypePn3t ? 5 : 4);
    if (!rw_forced) cfg.rw = 4;
    if (cfg.rw != 2 && cfg.rw != 4) return cudaErrorInvalidValue;
    if (cfg.cb <= 0) cfg.cb = nv ? 2 : 8;
    if (!nv && cfg.cb % 8 != 0) return cudaErrorInvalidValue;
    if (!ns_forced) cfg.ns = 4;
    const int sms = device_sm_count();
    const uint32_t bfrag_per_unit = 64u * a.M * steps;
    const int s_cap = std::min(16, U);
    if (!s_forced) {
        // Smallest cluster that keeps x and its fragments within budget, then widen (up to the
        // portable 8) while the grid is short of two CTAs per SM.
        const uint32_t budget = 48 * 1024;
        const int G = static_cast<int>((N + 16 * cfg.rw - 1) / (16 * cfg.rw));
        int S = 1;
        const uint32_t x_per_unit = static_cast<uint32_t>(a.M) * (nv ? 256 * 2 : (type == kTypePn3t ? 80 : 64) * 4);
        auto bytes_for = [&](int s) { return (bfrag_per_unit + x_per_unit) * align_units * ((U + s - 1) / s); };
        while (S < 8 && S < U && bytes_for(S) > budget) ++S;
        while (S < 8 && S < U && static_cast<int64_t>(G) * S < 2LL * sms) ++S;
        cfg.S = S;
    }
    cfg.S = std::max(1, std::min(cfg.S, s_cap));
    // Shrink until the shared-memory map fits: fewer stages, then fewer row warps, then a
    // wider (non-portable, up to 16) cluster.
    const int unit_k = nv ? 256 : (type == kTypePn3t ? 80 : 64);
    const int x_bytes = nv ? 2 : 4;
    auto total_for = [&](int S, int rw, int ns) {
        const int units_max = align_units * ((U + S - 1) / S);
        return make_layout(nv, steps, a.M, units_max, unit_k, x_bytes, 16 * rw, cfg.cb, ns).total;
    };
    while (total_for(cfg.S, cfg.rw, cfg.ns) > 227u * 1024u) {
        if (!ns_forced && cfg.ns > 2) --cfg.ns;
        else if (!rw_forced && cfg.rw == 4) cfg.rw = 2;
        else if (!s_forced && cfg.S < s_cap) ++cfg.S;
        else return cudaErrorNotSupported;
    }
    const int R = 16 * cfg.rw;
    const int64_t G64 = (N + R - 1) / R;
    if (G64 > 65535) return cudaErrorNotSupported;
    const int G = static_cast<int>(G64);
    a.S = cfg.S;
    a.NS = cfg.ns;
    a.chunk = cfg.cb;
    const uint32_t total = total_for(cfg.S, cfg.rw, cfg.ns);
    if (type == kTypePn3t)
        return cfg.rw == 4 ? launch_nt<kTypePn3t, 4>(a, G, total, stream) : launch_nt<kTypePn3t, 2>(a, G, total, stream);
    if (type == kTypePn4t)
        return cfg.rw == 4 ? launch_nt<kTypePn4t, 4>(a, G, total, stream) : launch_nt<kTypePn4t, 2>(a, G, total, stream);
    return cfg.rw == 4 ? launch_nt<kTypeNvfp4, 4>(a, G, total, stream) : launch_nt<kTypeNvfp4, 2>(a, G, total, stream);
}

}  // namespace

cudaError_t launch_pn_gemv_mma(int type, const uint8_t* W, int64_t N, int64_t K, const float* X, int M, float* Y,
                               int* err, MmaConfig cfg, cudaStream_t stream) {
    if (N == 0) return cudaSuccess;
    const int blk = (type == kTypePn3t) ? 80 : 64;
    if (K / blk > INT32_MAX / 256 || M < 1 || M > kMaxM) return cudaErrorNotSupported;
    Args a{};
    a.W = W;
    a.scales = nullptr;
    a.X = X;
    a.Y = Y;
    a.err = err;
    a.g = 1.0f;
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.units = static_cast<int>(K / blk);
    a.M = M;
    if (a.units % 8 != 0) return cudaErrorNotSupported;
    return launch_common(type, a, N, cfg, stream);
}

cudaError_t launch_nvfp4_gemv_mma(const Nvfp4View& w, int64_t N, int64_t K, const uint16_t* X, int M, float* Y,
                                  int* err, MmaConfig cfg, cudaStream_t stream) {
    if (N == 0) return cudaSuccess;
    if (K % 256 != 0 || K > INT32_MAX / 32 || M < 1 || M > kMaxM) return cudaErrorNotSupported;
    Args a{};
    a.W = w.codes;
    a.scales = w.scales;
    a.X = X;
    a.Y = Y;
    a.err = err;
    a.g = w.g;
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.units = static_cast<int>(K / 256);
    a.M = M;
    return launch_common(kTypeNvfp4, a, N, cfg, stream);
}

}  // namespace pnq
