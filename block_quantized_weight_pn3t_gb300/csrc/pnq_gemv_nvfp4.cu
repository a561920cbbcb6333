// pnq_gemv_nvfp4.cu -- tensor-core NVFP4 (W4A16) GEMV straight from the packed weights (fast path).
// (The kernel template below also carries the PN decode of an earlier design; only the NVFP4
// instantiation is launched, the PN fast path lives in pnq_gemv_pn.cu.)
//
// What it computes: Y[m][n] = sum_k w[n][k] x[m][k] for 1 <= M <= 16, w decoded in registers
// just before the multiply ("PN weight format", sections Block layout and Value; TandemLLM
// "Quantisation and profiles", section NVFP4: unpack 4-bit codes to 16-bit numbers in
// registers and multiply on the tensor cores).
//
// Structure:
//  * Persistent grid, one wave: clusters of S CTAs (S = 1, 2, 4 or 8), one CTA per SM. The
//    weight rows are cut into 16-row tiles and each cluster owns a balanced contiguous range
//    of tiles; CTA rank q of a cluster owns the q-th slice of K. A cluster streams its tiles
//    in passes of TP tiles.
//  * In a CTA, one producer warp streams rows HBM -> shared memory with 1-D bulk copies (one
//    per row per stage; a stage row is 8 PN blocks = 272 = 17 x 16 bytes, or 512 NVFP4
//    weights) into an NS-stage ring guarded by mbarriers, L2 policy evict-first. RW consumer
//    warps split every stage along K (each takes its own blocks of the chunk for all tiles of
//    the pass), so any number of rows keeps every warp busy and each block's B fragments
//    feed TP independent mma chains. At the end of a pass the warps reduce through shared
//    memory; with S > 1 the CTAs of the cluster then exchange their partial rows through
//    distributed shared memory (ready / consumed mbarrier handshakes, double-buffered by
//    pass, summed in rank order: deterministic, no atomics, no global scratch).
//  * At start the producer also copies the CTA's slice of x into the last stages of the ring;
//    the consumers turn it into mma B fragments and release those stages for weights. x is
//    scaled by a power of two 2^sigma chosen per CTA and activation row from max|x| (so any
//    finite magnitude fits fp16) and split into fp16 hi + lo parts (about 22 bits), one mma
//    column each: M rows use 2M columns, NT = ceil(2M/8) n8 tiles.
//  * Decode: a 32-bit word gives two codes at the same shift in its two 16-bit halves, so one
//    LOP3 builds an f16x2 of (1024 + n) and one HADD2/HFMA2 makes it exactly n - z: an mma A
//    register with no conversion. Within a block the k order is free (x is permuted the
//    same way), which lets 2-byte aligned words be read as aligned words pairing the high
//    half of word i-1 with the low half of word i. Each block's mma sum is scaled once by
//    fp32(d). NVFP4 folds the E4M3FN group scale into A with one HMUL2 (e2m1 * e4m3 is exact
//    in fp16) and applies the global multiplier at the end.
//  * Programmatic dependent launch: every CTA lets the next grid in the stream start
//    launching, and no global data is read before the previous grid has completed (or, with
//    the static-weights option, only the weights, which the caller declares unchanged).
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
constexpr int kPnChunk = 8;   // PN blocks per stage row: 272 bytes, a multiple of 16
constexpr int kNvChunk = 2;   // NVFP4 256-weight units per stage row: 256 code + 32 scale bytes
constexpr int kNvSteps = 16;  // mma k16 steps per NVFP4 unit

__host__ __device__ constexpr uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// Shared-memory map, computed identically on host and device.
struct Layout {
    uint32_t bar_off;      // full[NS], empty[NS], x_ready, x_free, red_full[2], red_free[2]
    uint32_t misc_off;     // maxbits[16] u32, sig_in[16] f32, sig_out[16] f32, issued u32
    uint32_t red_off;      // [RW][TP][NT][32][4] f32 per-warp partial sums of a pass
    uint32_t part_off;     // [2][TP*16][M] f32 partial rows exchanged in the cluster (S > 1)
    uint32_t bfrag_off;    // B fragments of the CTA's K slice
    uint32_t bfrag_unit;   // bytes of B fragments per block (PN) / 256-weight unit (NVFP4)
    uint32_t stage_off;    // NS stages
    uint32_t stage_bytes;  // bytes per stage
    uint32_t pitch;        // bytes per row in a stage (codes for NVFP4)
    uint32_t pitch_s;      // NVFP4: bytes per row of the stage's scale area
    uint32_t scale_off;    // NVFP4: offset of the scale area inside a stage
    uint32_t x_stage;      // x is staged in stages [x_stage, NS) at start
    uint32_t total;
};

// Stage pitch: a multiple of 16 bytes whose quotient by 16 is odd, so the 8 row groups of
// a warp fall on distinct 16-byte bank groups.
__host__ __device__ constexpr uint32_t odd16_pitch(uint32_t bytes) {
    return ((align_up(bytes, 16) / 16) % 2 == 1) ? align_up(bytes, 16) : align_up(bytes, 16) + 16;
}

// unit_k: weights per unit (BLK for PN, 256 for NVFP4); x_bytes: bytes per x element;
// RW consumer warps, TP tiles of 16 rows per pass, NT n8 tiles.
__host__ __device__ inline Layout make_layout(bool nvfp4, int steps_per_unit, int M, int units_max, int unit_k,
                                              int x_bytes, int RW, int TP, int NT, int NS, int S) {
    Layout L{};
    const int R = 16 * TP;
    L.bar_off = 0;
    L.misc_off = align_up(8u * (2 * NS + 6), 16);
    L.red_off = L.misc_off + 256;
    L.part_off = align_up(L.red_off + 4u * RW * TP * NT * 32 * 4, 16);
    const uint32_t part_bytes = (S > 1) ? 2u * 4u * R * M : 0u;
    L.bfrag_off = align_up(L.part_off + part_bytes, 128);
    L.bfrag_unit = 64u * M * steps_per_unit;  // 8M lanes x steps x 8 bytes
    L.stage_off = align_up(L.bfrag_off + L.bfrag_unit * units_max, 128);
    if (!nvfp4) {
        L.pitch = odd16_pitch(34u * kPnChunk);
        L.pitch_s = 0;
        L.scale_off = 0;
        L.stage_bytes = align_up(L.pitch * R, 128);
    } else {
        L.pitch = odd16_pitch(128u * kNvChunk);
        L.pitch_s = odd16_pitch(16u * kNvChunk);
        L.scale_off = align_up(L.pitch * R, 128);
        L.stage_bytes = align_up(L.scale_off + L.pitch_s * R, 128);
    }
    const uint32_t xbytes = static_cast<uint32_t>(M) * units_max * unit_k * x_bytes;
    const uint32_t xst = (xbytes + L.stage_bytes - 1) / L.stage_bytes;
    L.x_stage = (xst >= static_cast<uint32_t>(NS)) ? 0u : NS - xst;  // 0 = does not fit (host rejects)
    L.total = L.stage_off + L.stage_bytes * NS;
    return L;
}

enum ArgFlags : int { kStaticWeights = 1 };

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
    int flags;              // ArgFlags
};

// ---- per-CTA work ----------------------------------------------------------------------

struct Slice {
    int u0;       // first unit of this CTA's K slice
    int nunits;   // units in the slice
    int nchunks;  // stage chunks per pass
};

__device__ __forceinline__ Slice cta_slice(const Args& a, uint32_t rank, int align_units, int chunk) {
    // Split units into S slices, each a multiple of align_units (8 blocks for PN so that a
    // stage row is a whole number of 16-byte lines).
    const int U = a.units / align_units;
    const int g0 = static_cast<int>((static_cast<int64_t>(rank) * U) / a.S);
    const int g1 = static_cast<int>((static_cast<int64_t>(rank + 1) * U) / a.S);
    Slice s;
    s.u0 = g0 * align_units;
    s.nunits = (g1 - g0) * align_units;
    s.nchunks = (s.nunits + chunk - 1) / chunk;
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
__device__ void compute_sigma(const Args& a, const uint8_t* xs, int klen, uint8_t* smem, const Layout& L, int nct) {
    uint32_t* maxbits = reinterpret_cast<uint32_t*>(smem + L.misc_off);
    float* sig_in = reinterpret_cast<float*>(smem + L.misc_off + 64);
    float* sig_out = reinterpret_cast<float*>(smem + L.misc_off + 128);
    const int tid = threadIdx.x;
    const uint4* xv = reinterpret_cast<const uint4*>(xs);
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

// B fragment layout of one unit: for each n8 tile t, lanes 0..LU-1 (LU = lanes whose column
// is in use) hold 2 registers per mma step; steps are grouped in pairs as 16-byte records
// [pair q][lane], and an odd last step as 8-byte records [lane].
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
__device__ __forceinline__ void load_bfrag(const uint8_t* ubase, int M, int t, int lane, uint32_t (&b)[STEPS][2]) {
    const int LU = min(32, 8 * M - 32 * t);
    if (lane < LU) {
        const uint8_t* base = ubase + t * (256 * STEPS);
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

template <int TYPE>
__device__ void pn_fill_bfrag(const Args& a, const Slice& sl, const uint8_t* xs, uint8_t* smem, const Layout& L,
                              int nct) {
    using F = PnFmt<TYPE>;
    constexpr int STEPS = F::PAIRS;
    const float* sig_in = reinterpret_cast<const float*>(smem + L.misc_off + 64);
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

// One PN block for the first `tiles` of TP tiles x 16 rows: rowp[tile][0] = row g, [1] = row g + 8.
template <int TYPE, int NT, int TP, int ODD>
__device__ __forceinline__ void pn_block(const uint8_t* const (&rowp)[TP][2], int off, const uint8_t* ubase, int M,
                                         int lane, int tiles, float (&acc)[TP][NT][4]) {
    using F = PnFmt<TYPE>;
    constexpr int STEPS = F::PAIRS;
    const int tig = lane & 3;
    float d[TP][2];
    uint32_t wa[TP][2], wb[TP][2];
#pragma unroll
    for (int tp = 0; tp < TP; ++tp) {
        if (tp < tiles) {
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
    uint32_t b[NT][STEPS][2];
#pragma unroll
    for (int t = 0; t < NT; ++t) load_bfrag<STEPS>(ubase, M, t, lane, b[t]);
    float c[TP][NT][4];
#pragma unroll
    for (int tp = 0; tp < TP; ++tp)
#pragma unroll
        for (int t = 0; t < NT; ++t) c[tp][t][0] = c[tp][t][1] = c[tp][t][2] = c[tp][t][3] = 0.0f;
#define PNQ_STEP(J)                                                                                           \
    {                                                                                                         \
        _Pragma("unroll") for (int tp = 0; tp < TP; ++tp) {                                                   \
            if (tp < tiles) {                                                                                 \
                const uint32_t a0 = pn_pair<TYPE, J>(wa[tp][0]), a1 = pn_pair<TYPE, J>(wa[tp][1]);            \
                const uint32_t a2 = pn_pair<TYPE, J>(wb[tp][0]), a3 = pn_pair<TYPE, J>(wb[tp][1]);            \
                _Pragma("unroll") for (int t = 0; t < NT; ++t)                                                \
                    mma_f16_16816(c[tp][t], a0, a1, a2, a3, b[t][J][0], b[t][J][1]);                           \
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
    for (int tp = 0; tp < TP; ++tp) {
        if (tp < tiles) {
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                acc[tp][t][0] = fmaf(d[tp][0], c[tp][t][0], acc[tp][t][0]);
                acc[tp][t][1] = fmaf(d[tp][0], c[tp][t][1], acc[tp][t][1]);
                acc[tp][t][2] = fmaf(d[tp][1], c[tp][t][2], acc[tp][t][2]);
                acc[tp][t][3] = fmaf(d[tp][1], c[tp][t][3], acc[tp][t][3]);
            }
        }
    }
}

// ---- NVFP4 decode --------------------------------------------------------------------------
// A 256-weight unit of one row is 32 code words (8 codes each, one 16-weight group per two
// words) and 16 scale bytes. Lane tig owns words tig + 4q (q = 0..7). Step (q2, i) uses byte
// i of words tig + 8 q2 (A registers 0, 1) and tig + 8 q2 + 4 (registers 2, 3); a byte is
// the pair (k, k + 1) with k = 8 * word + 2 i.

__device__ __forceinline__ int nv_elem(int tig, int st, int r, int hi) {
    const int q2 = st >> 2, i = st & 3;
    return 8 * (tig + 8 * q2 + 4 * r) + 2 * i + hi;
}

__device__ void nv_fill_bfrag(const Args& a, const Slice& sl, const uint8_t* xs, uint8_t* smem, const Layout& L,
                              int nct) {
    const float* sig_in = reinterpret_cast<const float*>(smem + L.misc_off + 64);
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

// Groups q2 in [Q0, Q0 + NQ) of one NVFP4 unit for the first `tiles` of TP tiles:
// cp[tile][h] = codes of row (g, g + 8), sp[tile][h] = its scales.
template <int NT, int TP, int NQ>
__device__ __forceinline__ void nv_unit(const uint8_t* const (&cp)[TP][2], const uint8_t* const (&sp)[TP][2],
                                        int coff, int soff, const uint8_t* ubase, int M, int lane, int tiles, int Q0,
                                        float (&acc)[TP][NT][4]) {
    const int tig = lane & 3;
    const uint32_t ssel = (tig >> 1) | (((tig >> 1) + 2) << 4);  // bytes tig/2 and tig/2 + 2
#pragma unroll
    for (int qq = 0; qq < NQ; ++qq) {
        const int q2 = Q0 + qq;
        uint32_t b[NT][4][2];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int LU = min(32, 8 * M - 32 * t);
            if (lane < LU) {
                const uint8_t* base = ubase + t * (256 * kNvSteps);
                const uint4 v0 = *reinterpret_cast<const uint4*>(base + (2 * q2) * LU * 16 + lane * 16);
                const uint4 v1 = *reinterpret_cast<const uint4*>(base + (2 * q2 + 1) * LU * 16 + lane * 16);
                b[t][0][0] = v0.x; b[t][0][1] = v0.y; b[t][1][0] = v0.z; b[t][1][1] = v0.w;
                b[t][2][0] = v1.x; b[t][2][1] = v1.y; b[t][3][0] = v1.z; b[t][3][1] = v1.w;
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) b[t][i][0] = b[t][i][1] = 0u;
            }
        }
#pragma unroll
        for (int tp = 0; tp < TP; ++tp) {
            if (tp >= tiles) continue;
            const uint8_t* c0 = cp[tp][0] + coff;
            const uint8_t* c1 = cp[tp][1] + coff;
            const uint32_t w0a = *reinterpret_cast<const uint32_t*>(c0 + 4 * (tig + 8 * q2));
            const uint32_t w0b = *reinterpret_cast<const uint32_t*>(c0 + 4 * (tig + 8 * q2 + 4));
            const uint32_t w1a = *reinterpret_cast<const uint32_t*>(c1 + 4 * (tig + 8 * q2));
            const uint32_t w1b = *reinterpret_cast<const uint32_t*>(c1 + 4 * (tig + 8 * q2 + 4));
            // scales of groups 4 q2 + tig/2 (words tig + 8 q2) and 4 q2 + 2 + tig/2 (+4)
            const uint32_t sc0 =
                e4m3x2_to_f16x2(prmt(*reinterpret_cast<const uint32_t*>(sp[tp][0] + soff + 4 * q2), 0u, ssel));
            const uint32_t sc1 =
                e4m3x2_to_f16x2(prmt(*reinterpret_cast<const uint32_t*>(sp[tp][1] + soff + 4 * q2), 0u, ssel));
            const uint32_t s0a = prmt(sc0, sc0, 0x1010u), s0b = prmt(sc0, sc0, 0x3232u);
            const uint32_t s1a = prmt(sc1, sc1, 0x1010u), s1b = prmt(sc1, sc1, 0x3232u);
#define PNQ_NVSTEP(I)                                                                                       \
    {                                                                                                       \
        const uint32_t a0 = hmul2_u32(e2m1x2_to_f16x2<I>(w0a), s0a);                                        \
        const uint32_t a1 = hmul2_u32(e2m1x2_to_f16x2<I>(w1a), s1a);                                        \
        const uint32_t a2 = hmul2_u32(e2m1x2_to_f16x2<I>(w0b), s0b);                                        \
        const uint32_t a3 = hmul2_u32(e2m1x2_to_f16x2<I>(w1b), s1b);                                        \
        _Pragma("unroll") for (int t = 0; t < NT; ++t)                                                      \
            mma_f16_16816(acc[tp][t], a0, a1, a2, a3, b[t][I][0], b[t][I][1]);                               \
    }
            PNQ_NVSTEP(0)
            PNQ_NVSTEP(1)
            PNQ_NVSTEP(2)
            PNQ_NVSTEP(3)
#undef PNQ_NVSTEP
        }
    }
}


// ---- the kernel ---------------------------------------------------------------------------------

template <int TYPE, int NT, int RW>
__global__ void __launch_bounds__(32 * (RW + 1), 1) gemv_mma_kernel(const Args a) {
    constexpr bool kNv = (TYPE == kTypeNvfp4);
    constexpr int TP = RW;  // 16-row tiles per pass; after a pass warp w reduces tile w
    constexpr int R = 16 * TP;
    constexpr int kPnType = kNv ? kTypePn4t : TYPE;
    constexpr int kSteps = kNv ? kNvSteps : PnFmt<kPnType>::PAIRS;
    constexpr int kAlignUnits = kNv ? 1 : 8;
    constexpr int kChunk = kNv ? kNvChunk : kPnChunk;
    constexpr int kUnitK = kNv ? 256 : PnFmt<kPnType>::BLK;
    constexpr int kXBytes = kNv ? 2 : 4;
    constexpr int kBlkPerWarp = kPnChunk / RW;  // PN blocks of a chunk per warp (even)
    constexpr int kQPerWarp = 4 / RW;           // NVFP4 step groups of a unit per warp
    extern __shared__ __align__(128) uint8_t smem[];

    const uint32_t rank = (a.S > 1) ? cluster_ctarank() : 0u;
    const int units_max = kAlignUnits * ((a.units / kAlignUnits + a.S - 1) / a.S);
    const Layout L = make_layout(kNv, kSteps, a.M, units_max, kUnitK, kXBytes, RW, TP, NT, a.NS, a.S);
    const Slice sl = cta_slice(a, rank, kAlignUnits, kChunk);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // this cluster's tiles: a balanced contiguous share of the 16-row tiles
    const int T16 = (a.N + 15) / 16;
    const int cl = blockIdx.y, ncl = gridDim.y;
    const int t_begin = static_cast<int>((static_cast<int64_t>(cl) * T16) / ncl);
    const int t_end = static_cast<int>((static_cast<int64_t>(cl + 1) * T16) / ncl);
    const int npasses = (t_end - t_begin + TP - 1) / TP;
    const int total_chunks = npasses * sl.nchunks;

    const uint32_t bar0 = smem_addr(smem + L.bar_off);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (a.NS + s); };
    const uint32_t x_ready = bar0 + 8u * (2 * a.NS);
    const uint32_t x_free = bar0 + 8u * (2 * a.NS + 1);
    auto red_full = [&](int b) { return bar0 + 8u * (2 * a.NS + 2 + b); };
    auto red_free = [&](int b) { return bar0 + 8u * (2 * a.NS + 4 + b); };
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L.misc_off);
    uint8_t* xs = smem + L.stage_off + L.x_stage * L.stage_bytes;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.NS; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), RW);
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
    if (threadIdx.x < 16) misc[threadIdx.x] = 0u;  // maxbits
    if (threadIdx.x == 16) misc[48] = 0u;          // issued
    __syncthreads();
    if (a.S > 1) cluster_sync();  // every CTA's barriers exist before any remote arrive

    if (warp == RW) {
        // ---------------- producer warp ----------------
        const uint64_t pol = l2_policy_evict_first();
        const size_t rowc = kNv ? static_cast<size_t>(a.K) / 2 : static_cast<size_t>(a.units) * kBlockBytes;
        const size_t rows_ = static_cast<size_t>(a.K) / 16;
        bool ok = true;
        auto issue = [&](int gch) {
            const int p = gch / sl.nchunks, c = gch - p * sl.nchunks;
            const int s = gch % a.NS;
            if (gch >= a.NS) {
                if (!mbar_wait_bounded(empty_bar(s), ((gch / a.NS) - 1) & 1)) return false;
            } else if (s >= static_cast<int>(L.x_stage)) {
                if (!mbar_wait_bounded(x_free, 0)) return false;
            }
            const int t0 = t_begin + p * TP;
            const int rbase = 16 * t0;
            const int rows_valid = min(16 * min(TP, t_end - t0), a.N - rbase);
            const int n_in = min(kChunk, sl.nunits - c * kChunk);
            const uint32_t dst = smem_addr(smem + L.stage_off + s * L.stage_bytes);
            if (!kNv) {
                const uint32_t bytes = static_cast<uint32_t>(n_in * kBlockBytes);
                if (lane == 0) mbar_arrive_expect_tx(full_bar(s), bytes * rows_valid);
                __syncwarp();
                const uint8_t* src = a.W + static_cast<size_t>(rbase) * rowc +
                                     static_cast<size_t>(sl.u0 + c * kChunk) * kBlockBytes;
                for (int r = lane; r < rows_valid; r += 32)
                    bulk_g2s(dst + r * L.pitch, src + r * rowc, bytes, full_bar(s), pol);
            } else {
                const uint32_t cbytes = 128u * n_in, sbytes = 16u * n_in;
                if (lane == 0) mbar_arrive_expect_tx(full_bar(s), (cbytes + sbytes) * rows_valid);
                __syncwarp();
                const uint8_t* c0 = a.W + static_cast<size_t>(rbase) * rowc + static_cast<size_t>(sl.u0 + c * kChunk) * 128;
                const uint8_t* s0 =
                    a.scales + static_cast<size_t>(rbase) * rows_ + static_cast<size_t>(sl.u0 + c * kChunk) * 16;
                for (int r = lane; r < rows_valid; r += 32) {
                    bulk_g2s(dst + r * L.pitch, c0 + r * rowc, cbytes, full_bar(s), pol);
                    bulk_g2s(dst + L.scale_off + r * L.pitch_s, s0 + r * rows_, sbytes, full_bar(s), pol);
                }
            }
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
            // the CTA's slice of x: one bulk copy per activation row (16-byte aligned: X is, and
            // the slice starts at a multiple of 64 elements)
            const uint32_t xbytes = static_cast<uint32_t>(sl.nunits * kUnitK * kXBytes);
            if (lane == 0) mbar_arrive_expect_tx(x_ready, xbytes * a.M);
            __syncwarp();
            const uint8_t* xsrc = static_cast<const uint8_t*>(a.X) + static_cast<size_t>(sl.u0) * kUnitK * kXBytes;
            if (lane < a.M)
                bulk_g2s_plain(smem_addr(xs) + lane * xbytes, xsrc + static_cast<size_t>(lane) * a.K * kXBytes, xbytes,
                               x_ready);
        }
        for (; ok && gch < total_chunks; ++gch) ok = issue(gch);
        if (!ok && lane == 0) record_error(a.err, kErrEmptyWait);
        if (lane == 0) misc[48] = static_cast<uint32_t>(ok ? total_chunks : gch);
    } else {
        // ---------------- consumer warps ----------------
        const int nct = 32 * RW;
        const int klen = sl.nunits * kUnitK;
        if (!mbar_wait_bounded(x_ready, 0) && lane == 0) record_error(a.err, kErrFullWait);
        compute_sigma<kNv>(a, xs, klen, smem, L, nct);
        if constexpr (kNv)
            nv_fill_bfrag(a, sl, xs, smem, L, nct);
        else
            pn_fill_bfrag<TYPE>(a, sl, xs, smem, L, nct);
        named_sync(1, nct);
        if (threadIdx.x == 0) mbar_arrive(x_free);  // the x stages may now take weights

        const int g = lane >> 2, tig = lane & 3;
        const float* sig_out = reinterpret_cast<const float*>(smem + L.misc_off + 128);
        float* red = reinterpret_cast<float*>(smem + L.red_off);
        const uint32_t part_addr = smem_addr(smem + L.part_off);
        const uint32_t part_stride = 4u * R * a.M;  // bytes per pass buffer
        bool ok = true;
        int p = 0;
        for (; p < npasses && ok; ++p) {
            const int t0 = t_begin + p * TP;
            const int tiles = min(TP, t_end - t0);
            const int rbase = 16 * t0;
            float acc[TP][NT][4];
#pragma unroll
            for (int tp = 0; tp < TP; ++tp)
#pragma unroll
                for (int t = 0; t < NT; ++t) acc[tp][t][0] = acc[tp][t][1] = acc[tp][t][2] = acc[tp][t][3] = 0.0f;
            for (int c = 0; c < sl.nchunks; ++c) {
                const int gch = p * sl.nchunks + c;
                const int s = gch % a.NS;
                if (!mbar_wait_bounded(full_bar(s), (gch / a.NS) & 1)) {
                    if (lane == 0) record_error(a.err, kErrFullWait);
                    ok = false;
                    break;
                }
                const uint8_t* st = smem + L.stage_off + s * L.stage_bytes;
                const uint8_t* ubase0 = smem + L.bfrag_off + (c * kChunk) * L.bfrag_unit;
                if constexpr (!kNv) {
                    const uint8_t* rowp[TP][2];
#pragma unroll
                    for (int tp = 0; tp < TP; ++tp) {
                        rowp[tp][0] = st + (16 * tp + g) * L.pitch;
                        rowp[tp][1] = rowp[tp][0] + 8 * L.pitch;
                    }
                    // PN slices are whole chunks; this warp takes blocks [warp * kBlkPerWarp, +kBlkPerWarp)
#pragma unroll
                    for (int j = 0; j < kBlkPerWarp; j += 2) {
                        const int bl = warp * kBlkPerWarp + j;
                        pn_block<TYPE, NT, TP, 0>(rowp, kBlockBytes * bl, ubase0 + bl * L.bfrag_unit, a.M, lane, tiles,
                                                  acc);
                        pn_block<TYPE, NT, TP, 1>(rowp, kBlockBytes * (bl + 1), ubase0 + (bl + 1) * L.bfrag_unit, a.M,
                                                  lane, tiles, acc);
                    }
                } else {
                    const uint8_t* cp[TP][2];
                    const uint8_t* sp[TP][2];
#pragma unroll
                    for (int tp = 0; tp < TP; ++tp) {
                        const int r = 16 * tp + g;
                        cp[tp][0] = st + r * L.pitch;
                        cp[tp][1] = cp[tp][0] + 8 * L.pitch;
                        sp[tp][0] = st + L.scale_off + r * L.pitch_s;
                        sp[tp][1] = sp[tp][0] + 8 * L.pitch_s;
                    }
                    const int n_in = min(kChunk, sl.nunits - c * kChunk);
                    for (int u = 0; u < n_in; ++u)
                        nv_unit<NT, TP, kQPerWarp>(cp, sp, 128 * u, 16 * u, ubase0 + u * L.bfrag_unit, a.M, lane, tiles,
                                                   warp * kQPerWarp, acc);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty_bar(s));
            }
            if (!ok) break;

            // ---- reduce the warps' K shares, then (S > 1) the cluster's K slices
            const int b = p & 1;
#pragma unroll
            for (int tp = 0; tp < TP; ++tp)
                if (tp < tiles)
#pragma unroll
                    for (int t = 0; t < NT; ++t)
                        *reinterpret_cast<float4*>(red + ((((warp * TP + tp) * NT + t) * 32 + lane) * 4)) =
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
                for (int w = 0; w < RW; ++w)
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        const float4 v = *reinterpret_cast<const float4*>(red + ((((w * TP + warp) * NT + t) * 32 + lane) * 4));
                        sum[t][0] += v.x;
                        sum[t][1] += v.y;
                        sum[t][2] += v.z;
                        sum[t][3] += v.w;
                    }
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const int m = 4 * t + tig;
                    if (m < a.M) {
                        const float so = kNv ? sig_out[m] * a.g : sig_out[m];
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
    // Drain: no CTA leaves while a bulk copy it issued may still be writing its shared memory.
    if (warp == RW && lane == 0) {
        if (!mbar_wait_bounded(x_ready, 0)) record_error(a.err, kErrDrainWait);
        const int issued = static_cast<int>(misc[48]);
        for (int c = max(0, issued - a.NS); c < issued; ++c)
            if (!mbar_wait_bounded(full_bar(c % a.NS), (c / a.NS) & 1)) record_error(a.err, kErrDrainWait);
    }
    if (a.S > 1) cluster_sync();  // no CTA leaves while a peer may still address its shared memory
}

// ---- host side --------------------------------------------------------------------------------------

template <int TYPE, int NT, int RW>
cudaError_t prepare_kernel(int S, size_t smem_bytes) {
    auto kern = gemv_mma_kernel<TYPE, NT, RW>;
    // The shared-memory opt-in is raised once per device and size (not on every launch, and
    // so never while a stream is being captured after the first eager call).
    static size_t opted[64] = {};
    static bool wide[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (opted[dev] < smem_bytes) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_bytes));
        if (e != cudaSuccess) return e;
        opted[dev] = smem_bytes;
    }
    if (S > 8 && !wide[dev]) {  // clusters of 9..16 CTAs are a non-portable opt-in
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        wide[dev] = true;
    }
    return cudaSuccess;
}

// Co-resident clusters of S CTAs with this shared-memory size (cached per device, S, size).
template <int TYPE, int NT, int RW>
int resident_clusters(int S, size_t smem_bytes) {
    struct Entry { int dev, S; size_t smem; int n; };
    static Entry cache[64];
    static int used = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    for (int i = 0; i < used; ++i)
        if (cache[i].dev == dev && cache[i].S == S && cache[i].smem == smem_bytes) return cache[i].n;
    if (prepare_kernel<TYPE, NT, RW>(S, smem_bytes) != cudaSuccess) return 0;
    auto kern = gemv_mma_kernel<TYPE, NT, RW>;
    int n = 0;
    if (S == 1) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32 * (RW + 1), smem_bytes) != cudaSuccess)
            return 0;
        n = per_sm * device_sm_count();
    } else {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(S, 1024, 1);
        cfg.blockDim = dim3(32 * (RW + 1), 1, 1);
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

template <int TYPE, int NT, int RW>
cudaError_t launch_one(const Args& a, int clusters, size_t smem_bytes, cudaStream_t stream) {
    cudaError_t e = prepare_kernel<TYPE, NT, RW>(a.S, smem_bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(a.S, clusters, 1);
    cfg.blockDim = dim3(32 * (RW + 1), 1, 1);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = stream;
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
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, gemv_mma_kernel<TYPE, NT, RW>, a);
}

// Environment override "rw,S,_,ns" (any field 0 = automatic), read once; used by the tile
// sweeps of the benchmark tooling and by the configuration tests.
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

// Picks the cluster size and stage count, sizes the persistent grid, and launches.
template <int TYPE, int NT, int RW>
cudaError_t plan_and_launch(Args a, const MmaConfig& cfg, bool static_weights, cudaStream_t stream) {
    constexpr bool nv = (TYPE == kTypeNvfp4);
    constexpr int steps = nv ? kNvSteps : (TYPE == kTypePn3t ? 5 : 4);
    constexpr int unit_k = nv ? 256 : (TYPE == kTypePn3t ? 80 : 64);
    constexpr int x_bytes = nv ? 2 : 4;
    constexpr int align_units = nv ? 1 : 8;
    const int U = a.units / align_units;
    const int T16 = (a.N + 15) / 16;
    auto layout_for = [&](int S, int ns) {
        const int units_max = align_units * ((U + S - 1) / S);
        return make_layout(nv, steps, a.M, units_max, unit_k, x_bytes, RW, RW, NT, ns, S);
    };
    // stage count: the requested one, else the smallest >= 4 that leaves room for x
    auto stages_for = [&](int S) {
        if (cfg.ns > 0) return (layout_for(S, cfg.ns).total <= 227u * 1024u && layout_for(S, cfg.ns).x_stage >= 1) ? cfg.ns : 0;
        for (int ns = 4; ns <= 12; ++ns) {
            const Layout L = layout_for(S, ns);
            if (L.total > 227u * 1024u) return 0;
            if (L.x_stage >= 1) return ns;
        }
        return 0;
    };
    int best_S = 0, best_ns = 0, best_clusters = 0;
    int64_t best_cost = INT64_MAX;
    const int s_list[] = {1, 2, 4, 8, 16};
    int s_forced = 0;  // a requested cluster size, rounded down to the list and to U
    if (cfg.S > 0)
        for (int S : s_list)
            if (S <= std::min(cfg.S, U)) s_forced = S;
    for (int S : s_list) {
        if (S > U) break;
        if (s_forced > 0 && S != s_forced) continue;
        const int ns = stages_for(S);
        if (ns == 0) continue;
        const int resident = resident_clusters<TYPE, NT, RW>(S, layout_for(S, ns).total);
        if (resident < 1) continue;
        const int clusters = std::min(resident, T16);
        // makespan in (16-row tile x unit) work items of the busiest CTA, plus a per-pass cost
        const int64_t tiles = (T16 + clusters - 1) / clusters;
        const int64_t units = (U + S - 1) / S;
        const int64_t cost = tiles * units * 16 + ((tiles + RW - 1) / RW) * (S > 1 ? 24 : 8);
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
    a.flags = static_weights ? kStaticWeights : 0;
    return launch_one<TYPE, NT, RW>(a, best_clusters, layout_for(best_S, best_ns).total, stream);
}

template <int TYPE>
cudaError_t launch_typed(const Args& a, MmaConfig cfg, bool static_weights, cudaStream_t stream) {
    const int nt = (2 * a.M + 7) / 8;
    int rw = cfg.rw > 0 ? cfg.rw : (nt <= 2 ? 4 : 2);
    if (rw != 2 && rw != 4) return cudaErrorInvalidValue;
    if (nt <= 1) return rw == 4 ? plan_and_launch<TYPE, 1, 4>(a, cfg, static_weights, stream)
                                : plan_and_launch<TYPE, 1, 2>(a, cfg, static_weights, stream);
    if (nt <= 2) return rw == 4 ? plan_and_launch<TYPE, 2, 4>(a, cfg, static_weights, stream)
                                : plan_and_launch<TYPE, 2, 2>(a, cfg, static_weights, stream);
    return rw == 4 ? plan_and_launch<TYPE, 4, 4>(a, cfg, static_weights, stream)
                   : plan_and_launch<TYPE, 4, 2>(a, cfg, static_weights, stream);
}

cudaError_t launch_common(int type, Args a, MmaConfig cfg, bool static_weights, cudaStream_t stream) {
    const MmaConfig env = env_config();
    if (cfg.rw <= 0) cfg.rw = env.rw;
    if (cfg.S <= 0) cfg.S = env.S;
    if (cfg.ns <= 0) cfg.ns = env.ns;
    if (cfg.ns != 0 && (cfg.ns < 2 || cfg.ns > 16)) return cudaErrorInvalidValue;
    if (reinterpret_cast<uintptr_t>(a.X) % 16 != 0) return cudaErrorNotSupported;  // x slices are bulk-copied
    (void)type;
    return launch_typed<kTypeNvfp4>(a, cfg, static_weights, stream);
}

}  // namespace

cudaError_t launch_nvfp4_gemv_mma(const Nvfp4View& w, int64_t N, int64_t K, const uint16_t* X, int M, float* Y,
                                  int* err, MmaConfig cfg, bool static_weights, cudaStream_t stream) {
    if (N == 0) return cudaSuccess;
    if (N > INT32_MAX || K % 256 != 0 || K > INT32_MAX / 32 || M < 1 || M > kMaxM) return cudaErrorNotSupported;
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
    return launch_common(kTypeNvfp4, a, cfg, static_weights, stream);
}

}  // namespace pnq
