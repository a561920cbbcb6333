// pnq_gemv_nvfp4.cu -- NVFP4 (W4A16) GEMV on the tensor cores with mma.sync, sm_103a (fast path).
//
// Computes Y[m][n] = sum_k w[n][k] x[m][k] for 1 <= M <= 16 with w = e2m1(code) * e4m3(scale) * g
// ("Quantisation and profiles", NVFP4; tensor-formats page, NVFP4 / E2M1 / E4M3FN): codes two per
// byte, low nibble = even k, one E4M3FN scale per 16 weights along K, one fp32 global multiplier;
// x is bf16. The weights are decoded in registers just before the multiply. Two paths:
//   - M <= 8: the row stream of this file (nv_rows_kernel, below);
//   - M = 9..16, and M <= 8 shapes whose row plan does not fit in shared memory: the strip
//     pipeline (cluster work split, weight stream, operand builders, on-chip reduction) of
//     pnq_cluster.cuh, with this file's NVFP4 format policy, described next.
//
// Unit and stage. A K unit is 256 weights of a row: 128 code bytes and 16 scale bytes. An 8-row
// piece is two tensor-map copies: the codes (8 rows x 128 bytes, with the 128-byte swizzle:
// 16-byte chunk c of row r lands at chunk c ^ (r % 8), so the eight rows a warp reads at once fall
// in different banks) and the scales (8 rows x 16 bytes). A 64-row stage holds the codes of its 64
// rows (8 KB) and then their scales (1 KB).
//
// Decode and multiply. Lane (g, c) of a warp owns code words c, c + 4, c + 8, c + 12 of each half
// unit (16 words of 8 codes) for rows g and g + 8; each word holds 8 codes of one scale group. A
// byte (two codes) becomes an f16x2 A register with cvt.rn.f16x2.e2m1x2 and one HMUL2 by the
// group's scale (cvt.rn.f16x2.e4m3x2): the product of an e2m1 and an e4m3 value is exact in fp16.
// Byte b of words c + 8q and c + 8q + 4 are k16 slice 4q + b of the half. B column m holds the
// matching x pairs of activation row m times 2^sigma (per unit and row, so that max |x| * 2^sigma
// lies in [2^14, 2^15)): a bf16 value scaled so is exact in fp16 down to 2^-14 (8 significant bits
// < 11); below that it rounds at 2^-24, 2^-38 of the row's largest |x|. The two half units' even
// and odd slices form four mma chains per warp; each unit's sums are scaled by g * 2^-sigma.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <mutex>

#include "pnq_cluster.cuh"

namespace pnq {
namespace {

constexpr int kUnitK = 256;                                // weights of a row per K unit
constexpr int kCodeRow = kUnitK / 2;                       // code bytes of a row per unit (128)
constexpr int kScaleRow = kUnitK / 16;                     // scale bytes of a row per unit (16)
constexpr int kCodeStage = kStageRows * kCodeRow;          // 8192
constexpr int kNvStageBytes = kCodeStage + kStageRows * kScaleRow;  // 9216, a multiple of 1024
constexpr int kNvPieceTx = kPieceRows * (kCodeRow + kScaleRow);     // 1152

// B operands of activation row m for one K unit (one builder warp): sigma from the row's largest
// |x| over the unit, the 16-byte lane records (slices 2P and 2P + 1 in the lane of column m) and
// g * 2^-sigma. xr = the row's 256 bf16 x values in shared memory. Lane (P, c) = (lane / 4,
// lane % 4) builds the record of slices S = 2P, 2P + 1 (half S / 8, q = (S % 8) / 4, byte
// b = S % 4): register r holds the x pair at k = 8 * (16 * half + c + 8q + 4r) + 2b.
template <int NT>
__device__ __forceinline__ void nv_build_row(uint8_t* rec, float* so, const uint16_t* xr, int m, float g, int lane) {
    const uint4 xv = reinterpret_cast<const uint4*>(xr)[lane];
    const uint32_t w[4] = {xv.x, xv.y, xv.z, xv.w};
    uint32_t mx = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) mx = max(mx, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
    const uint32_t bits = __reduce_max_sync(0xffffffffu, mx) << 16;  // the fp32 bits of max |x|
    const int E = static_cast<int>(bits >> 23);
    int sg = (bits == 0 || E >= 255) ? 0 : 141 - E;  // max < 2^(E - 126)
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
    uint8_t* tb = rec + (m >> 3) * 4096 + P * 512;
    *reinterpret_cast<uint4*>(tb + ((((m & 7) << 2) | c) * 16)) = make_uint4(v[0], v[1], v[2], v[3]);
    if (lane == 0) so[m] = exp2i(-sg) * g;
}

// The NVFP4 format policy of the cluster pipeline.
template <int NT>
struct NvMma {
    static constexpr int MAPS = 4;  // codes, scales with 8-row boxes (pieces); the same with 64-row boxes (stages)
    struct Extra {
        float g;
    };
    static constexpr int NB = NT;  // builder warps
    static constexpr int THREADS = 32 * (kConsumerWarps + 1 + NB);
    static constexpr int MINB = (NT == 1) ? 2 : 1;
    static constexpr int UK = kUnitK, X_BYTES = 2;
    static constexpr int STAGE_BYTES = kNvStageBytes, PIECE_TX = kNvPieceTx;
    static constexpr int REC = NT * 4096;  // 16 slices x 32 lanes x 8 bytes per n8 tile
    static constexpr int ZB = 16;          // g * 2^-sigma per activation row
    static constexpr double GROUP_S = 0.15e-6;
    struct Lane {
        int g, c;
        uint32_t sel0, sel1;  // scale byte (2j + c / 2) % 4 twice, for j even / odd
        uint32_t boff[NT];    // this lane's B record in tile t (a live column's for absent rows)
        uint32_t chunk[8];    // byte offset of logical 16-byte chunk q of the lane's rows (swizzled) + 4c
        __device__ Lane(int l, int M)
            : g(l >> 2), c(l & 3), sel0(((l & 3) >> 1) * 0x11u), sel1((2 + ((l & 3) >> 1)) * 0x11u) {
#pragma unroll
            for (int t = 0; t < NT; ++t) boff[t] = static_cast<uint32_t>((4 * min(g, max(0, M - 1 - 8 * t)) + c) * 16);
#pragma unroll
            for (int q = 0; q < 8; ++q) chunk[q] = static_cast<uint32_t>(((q ^ g) << 4) + 4 * c);
        }
    };
    struct Acc {
        float v[NT][4];  // rows g, g + 8 x activation rows 8t + 2c, 8t + 2c + 1
    };
    static __device__ __forceinline__ void issue(const CUtensorMap* maps, uint32_t dst, int p, int u, int row,
                                                 uint32_t bar, uint64_t pol) {
        tma_load_2d(dst + p * kPieceRows * kCodeRow, &maps[0], u * (kCodeRow / 4), row, bar, pol);
        tma_load_2d(dst + kCodeStage + p * kPieceRows * kScaleRow, &maps[1], u * (kScaleRow / 4), row, bar, pol);
    }
    static __device__ __forceinline__ void issue_stage(const CUtensorMap* maps, uint32_t dst, int u, int row,
                                                       uint32_t bar, uint64_t pol) {
        tma_load_2d(dst, &maps[2], u * (kCodeRow / 4), row, bar, pol);
        tma_load_2d(dst + kCodeStage, &maps[3], u * (kScaleRow / 4), row, bar, pol);
    }
    static __device__ __forceinline__ void zero_half(uint8_t* stg, int lg, int lane) {
        uint32_t* zc = reinterpret_cast<uint32_t*>(stg + (lg * kGroupRows + 8) * kCodeRow);
        for (int i = lane; i < 8 * kCodeRow / 4; i += 32) zc[i] = 0u;
        uint32_t* zs = reinterpret_cast<uint32_t*>(stg + kCodeStage + (lg * kGroupRows + 8) * kScaleRow);
        for (int i = lane; i < 8 * kScaleRow / 4; i += 32) zs[i] = 0u;
    }
    static __device__ __forceinline__ void build(uint8_t* rec, float* zb, const uint8_t* xrow, int m, const Extra& e,
                                                 int lane) {
        nv_build_row<NT>(rec, zb, reinterpret_cast<const uint16_t*>(xrow), m, e.g, lane);
    }
    static __device__ __forceinline__ void group(const uint8_t* stg, int lg, const uint8_t* recu, const float*, int,
                                                 const Lane& ln, Acc& acc) {
        const uint32_t st = smem_addr(stg);
        const uint32_t srow = st + static_cast<uint32_t>((lg * kGroupRows + ln.g) * kCodeRow);  // rows g, g + 8
        const uint32_t sscl = st + kCodeStage + static_cast<uint32_t>((lg * kGroupRows + ln.g) * kScaleRow);
        const uint32_t rec_s = smem_addr(recu);
        uint32_t srec[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) srec[t] = rec_s + ln.boff[t];
        // code words c + 4j of each half H (swizzled 16-byte chunk 4H + j of the row) and the
        // group scales as f16x2
        uint32_t w[2][2][4], sc[2][2][4];
        static_for<2>([&](auto Hh) {
            constexpr int h = decltype(Hh)::value;
            const uint4 s4 = ld_shared_v4<h * 8 * kScaleRow>(sscl);
            static_for<2>([&](auto HH) {
                constexpr int H = decltype(HH)::value;
                static_for<4>([&](auto Jj) {
                    constexpr int j = decltype(Jj)::value;
                    w[H][h][j] = ld_shared_u32<h * 8 * kCodeRow>(srow + ln.chunk[4 * H + j]);
                });
                // word c + 4j is scale group 8H + 2j + c / 2: byte (2j + c / 2) % 4 of scale word 2H + j / 2
                const uint32_t sw0 = H ? s4.z : s4.x, sw1 = H ? s4.w : s4.y;
                sc[H][h][0] = e4m3x2_to_f16x2(prmt(sw0, 0u, ln.sel0));
                sc[H][h][1] = e4m3x2_to_f16x2(prmt(sw0, 0u, ln.sel1));
                sc[H][h][2] = e4m3x2_to_f16x2(prmt(sw1, 0u, ln.sel0));
                sc[H][h][3] = e4m3x2_to_f16x2(prmt(sw1, 0u, ln.sel1));
            });
        });
        float c2[2][2][NT][4];  // [half][slice parity][tile]
        uint4 bq[2][NT];        // B records of a pair of slices, per half
        static_for<8>([&](auto Sc) {
            constexpr int S = decltype(Sc)::value, q = S >> 2, bt = S & 3;
            static_for<2>([&](auto HH) {
                constexpr int H = decltype(HH)::value;
                if constexpr ((S & 1) == 0)
                    static_for<NT>([&](auto T) {
                        constexpr int t = decltype(T)::value;
                        bq[H][t] = ld_shared_v4<t * 4096 + (4 * H + (S >> 1)) * 512>(srec[t]);
                    });
                const uint32_t a0 = hmul2_u32(e2m1x2_to_f16x2<bt>(w[H][0][2 * q]), sc[H][0][2 * q]);
                const uint32_t a1 = hmul2_u32(e2m1x2_to_f16x2<bt>(w[H][1][2 * q]), sc[H][1][2 * q]);
                const uint32_t a2 = hmul2_u32(e2m1x2_to_f16x2<bt>(w[H][0][2 * q + 1]), sc[H][0][2 * q + 1]);
                const uint32_t a3 = hmul2_u32(e2m1x2_to_f16x2<bt>(w[H][1][2 * q + 1]), sc[H][1][2 * q + 1]);
                static_for<NT>([&](auto T) {
                    constexpr int t = decltype(T)::value;
                    const uint32_t b0 = (S & 1) ? bq[H][t].z : bq[H][t].x, b1 = (S & 1) ? bq[H][t].w : bq[H][t].y;
                    if constexpr (S < 2)
                        mma_f16_16816_z(c2[H][S & 1][t], a0, a1, a2, a3, b0, b1);
                    else
                        mma_f16_16816(c2[H][S & 1][t], a0, a1, a2, a3, b0, b1);
                });
            });
        });
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc.v[t][i] = (c2[0][0][t][i] + c2[0][1][t][i]) + (c2[1][0][t][i] + c2[1][1][t][i]);
    }
    // rows g, g + 8 of the group, activation rows 8t + 2c (+ 1): partial += sums * g * 2^-sigma
    static __device__ __forceinline__ void flush(float* part, int rc, int lr, const float* so, int M, const Lane& ln,
                                                 const Acc& acc) {
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int m = 8 * t + 2 * ln.c + i;
                if (m < M) {
                    const float f = so[m];
                    float* pr = part + m * rc + lr + ln.g;
                    pr[0] = fmaf(acc.v[t][i], f, pr[0]);
                    pr[8] = fmaf(acc.v[t][2 + i], f, pr[8]);
                }
            }
    }
};

// ---- row-stream path (M <= 8) ------------------------------------------------------------------
//
// The structure of the PN row stream (pnq_gemv_pn.cu): each CTA owns whole rows; a stage is a
// 16-row group of one K segment (all units of a short row, or a near-equal share of a long one),
// brought in by two 1-D bulk copies per row (its code bytes and its scale bytes), issued by two
// producer warps; rows are `pitch` bytes apart in each region, padded so that pitch / 16 is odd
// (the eight rows a warp reads at once then fall in different banks; no swizzle is needed). All
// of x (bf16 [M][K]) comes in with one bulk copy per activation row; the consumer warps build the
// B operands of every unit between them (records of the 4M lanes whose columns are live) and the
// (row group, unit) tasks of the stages are dealt to them in turn. Clusters of CL = 1, 2, 4 or 8
// CTAs may split K: CTA r of a cluster streams, builds and multiplies only units
// [r U / CL, (r + 1) U / CL) of the cluster's rows, and CTA r writes a share of the rows, adding
// every CTA's row sums in CTA order through distributed shared memory (deterministic).

constexpr int kNrWarps = 8;
constexpr int kNrProducers = 2;
constexpr int kNrThreads = 32 * (kNrWarps + kNrProducers);
constexpr int kNrMaxSeg = 32;
constexpr int kNrMaxStages = 8;
constexpr int kNrMaxM = 8;  // activation rows (one n8 tile: a column per row)
constexpr uint32_t kNrSmem = 226u * 1024u;
constexpr int nr_pitch(int bytes) { return ((bytes / 16) & 1) ? bytes : bytes + 16; }

// B operands of activation row m (m < LR / 4) for one unit, in the compact layout: slice pair P
// at P * LR * 16, lane record (4 (m) + c) * 16 within it.
template <int LR>
__device__ __forceinline__ void nv_build_row_compact(uint8_t* rec, float* so, const uint16_t* xr, int m, float g,
                                                     int lane) {
    const uint4 xv = reinterpret_cast<const uint4*>(xr)[lane];
    const uint32_t w[4] = {xv.x, xv.y, xv.z, xv.w};
    uint32_t mx = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) mx = max(mx, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
    const uint32_t bits = __reduce_max_sync(0xffffffffu, mx) << 16;
    const int E = static_cast<int>(bits >> 23);
    int sg = (bits == 0 || E >= 255) ? 0 : 141 - E;
    sg = min(100, max(-100, sg));
    const float si = exp2i(sg);
    const int P = lane >> 2, c = lane & 3;
    const uint32_t* x32 = reinterpret_cast<const uint32_t*>(xr);
    uint32_t v[4];
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
        const int S = 2 * P + (q4 >> 1), r = q4 & 1;
        const int half = S >> 3, q = (S >> 2) & 1, b = S & 3;
        const uint32_t pair = x32[4 * (16 * half + c + 8 * q + 4 * r) + b];
        v[q4] = f32x2_to_f16x2(__uint_as_float(pair << 16) * si, __uint_as_float(pair & 0xFFFF0000u) * si);
    }
    *reinterpret_cast<uint4*>(rec + P * (LR * 16) + ((m << 2) | c) * 16) = make_uint4(v[0], v[1], v[2], v[3]);
    if (lane == 0) so[m] = exp2i(-sg) * g;
}

// One (row group, unit) task: rows g (h = 0) and g + 8 (h = 1) at scode[h] (code bytes of the
// unit) and sscl[h] (its 16 scale bytes); srec = the lane's B record. acc: the four accumulators
// of the lane (rows g, g + 8 x columns 2c, 2c + 1), already summed over the unit's slices.
template <int LR>
__device__ __forceinline__ void nv_task(const uint32_t (&scode)[2], const uint32_t (&sscl)[2], uint32_t srec, int c,
                                        uint32_t sel0, uint32_t sel1, float (&acc)[4]) {
    uint32_t w[2][2][4], sc[2][2][4];
    static_for<2>([&](auto Hh) {
        constexpr int h = decltype(Hh)::value;
        const uint4 s4 = ld_shared_v4<0>(sscl[h]);
        static_for<2>([&](auto HH) {
            constexpr int H = decltype(HH)::value;
            static_for<4>([&](auto Jj) {
                constexpr int j = decltype(Jj)::value;
                w[H][h][j] = ld_shared_u32<(4 * H + j) * 16>(scode[h]);  // word c + 4j of half H (scode has + 4c)
            });
            const uint32_t sw0 = H ? s4.z : s4.x, sw1 = H ? s4.w : s4.y;
            sc[H][h][0] = e4m3x2_to_f16x2(prmt(sw0, 0u, sel0));
            sc[H][h][1] = e4m3x2_to_f16x2(prmt(sw0, 0u, sel1));
            sc[H][h][2] = e4m3x2_to_f16x2(prmt(sw1, 0u, sel0));
            sc[H][h][3] = e4m3x2_to_f16x2(prmt(sw1, 0u, sel1));
        });
    });
    float c2[2][2][4];
    uint4 bq[2];
    static_for<8>([&](auto Sc) {
        constexpr int S = decltype(Sc)::value, q = S >> 2, bt = S & 3;
        static_for<2>([&](auto HH) {
            constexpr int H = decltype(HH)::value;
            if constexpr ((S & 1) == 0) bq[H] = ld_shared_v4<(4 * H + (S >> 1)) * LR * 16>(srec);
            const uint32_t a0 = hmul2_u32(e2m1x2_to_f16x2<bt>(w[H][0][2 * q]), sc[H][0][2 * q]);
            const uint32_t a1 = hmul2_u32(e2m1x2_to_f16x2<bt>(w[H][1][2 * q]), sc[H][1][2 * q]);
            const uint32_t a2 = hmul2_u32(e2m1x2_to_f16x2<bt>(w[H][0][2 * q + 1]), sc[H][0][2 * q + 1]);
            const uint32_t a3 = hmul2_u32(e2m1x2_to_f16x2<bt>(w[H][1][2 * q + 1]), sc[H][1][2 * q + 1]);
            const uint32_t b0 = (S & 1) ? bq[H].z : bq[H].x, b1 = (S & 1) ? bq[H].w : bq[H].y;
            if constexpr (S < 2)
                mma_f16_16816_z(c2[H][S & 1], a0, a1, a2, a3, b0, b1);
            else
                mma_f16_16816(c2[H][S & 1], a0, a1, a2, a3, b0, b1);
        });
    });
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = (c2[0][0][i] + c2[0][1][i]) + (c2[1][0][i] + c2[1][1][i]);
}

struct NrArgs {
    const uint8_t* codes;
    const uint8_t* scales;
    const uint16_t* X;
    float* Y;
    int* err;
    float g;
    int N, K, M, U, G, S, nseg, rows_pad;
    int CL;  // CTAs of a cluster: CTA r of a cluster takes K units [r U / CL, (r + 1) U / CL) of its rows
    unsigned flags;
    uint32_t off_rec, off_so, off_x, off_part, off_stage, stage_bytes, scale_region;  // scale region offset in a stage
};

template <int LR>
__global__ void __launch_bounds__(kNrThreads, 1) nv_rows_kernel(const __grid_constant__ NrArgs a) {
    constexpr int REC = 8 * LR * 16;  // bytes of one unit's B records
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t bar0 = smem_addr(base);
    const int S = a.S, M = a.M, nseg = a.nseg;
    const int CL = a.CL, cr = static_cast<int>(blockIdx.x) % CL, cid = static_cast<int>(blockIdx.x) / CL;
    const int ua = cr * a.U / CL, U = (cr + 1) * a.U / CL - ua;  // this CTA's K units [ua, ua + U)
    const int xk = U * kUnitK;                                   // bf16 of an activation row it reads
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (S + s); };
    const uint32_t xfull = bar0 + 8u * (2 * S), xreq = bar0 + 8u * (2 * S + 1);
    auto stage = [&](int s) { return base + a.off_stage + static_cast<uint32_t>(s) * a.stage_bytes; };
    auto rec = [&](int u) { return base + a.off_rec + static_cast<uint32_t>(u) * REC; };
    auto so = [&](int u) { return reinterpret_cast<float*>(base + a.off_so) + u * kNrMaxM; };
    __shared__ int seg_tab[kNrMaxSeg + 1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r0 = static_cast<int64_t>(cid) * a.N / a.G, r1 = static_cast<int64_t>(cid + 1) * a.N / a.G;
    const int nrows = static_cast<int>(r1 - r0);
    const int nstages = (nrows + kGroupRows - 1) / kGroupRows * nseg;
    float* part = reinterpret_cast<float*>(base + a.off_part);  // [warp][m][rows_pad]
    const int64_t crow = a.K / 2, srow_b = a.K / 16;             // code / scale bytes per row

    if (threadIdx.x == 0) {
        griddep_launch_dependents();
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), kNrProducers);
            mbar_init(empty(s), kNrWarps);
        }
        for (int j = 0; j <= nseg; ++j) seg_tab[j] = j * U / nseg;
        mbar_init(xfull, 1);
        mbar_init(xreq, kNrWarps);
        mbar_fence_init();
    }
    __syncthreads();

    if (warp >= kNrWarps) {
        const int pr = (warp - kNrWarps) * 8;
        const uint64_t pol = l2_policy_evict_first();
        if (!(a.flags & kStaticWeights)) griddep_wait();
        bool ok = true;
        int s = 0;
        for (int i = 0, j = 0; s < nstages; ++s) {
            const int slot = s % S;
            if (s == 1 && !mbar_wait_warp(xreq, 0)) {  // x is requested before the ring fills
                ok = false;
                break;
            }
            if (s >= S && !mbar_wait_warp(empty(slot), ((s / S) - 1) & 1)) {
                ok = false;
                break;
            }
            const int mine = min(8, max(0, nrows - i * kGroupRows - pr));
            const int u0 = seg_tab[j], n = seg_tab[j + 1] - u0;
            const int cb = n * 128, sb = n * 16, pc = nr_pitch(cb), ps = nr_pitch(sb);
            if (lane == 0) mbar_arrive_expect_tx(full(slot), static_cast<uint32_t>(mine * (cb + sb)));
            __syncwarp();
            if (lane < mine) {
                const int64_t row = r0 + i * kGroupRows + pr + lane;
                const uint32_t dst = smem_addr(stage(slot));
                bulk_g2s(dst + static_cast<uint32_t>((pr + lane) * pc), a.codes + row * crow + (ua + u0) * 128,
                         static_cast<uint32_t>(cb), full(slot), pol);
                bulk_g2s(dst + a.scale_region + static_cast<uint32_t>((pr + lane) * ps),
                         a.scales + row * srow_b + (ua + u0) * 16, static_cast<uint32_t>(sb), full(slot), pol);
            }
            if (++j == nseg) {
                j = 0;
                ++i;
            }
        }
        if (!ok && lane == 0) record_error(a.err, kErrEmptyWait);
        bool drained = mbar_wait_warp(xfull, 0);
        for (int gg = max(0, s - S); drained && gg < s; ++gg) drained = mbar_wait_warp(full(gg % S), (gg / S) & 1);
        if (!drained && lane == 0) record_error(a.err, kErrDrainWait);
    } else {
        const int g = lane >> 2, c = lane & 3;
        const uint32_t sel0 = ((lane & 3) >> 1) * 0x11u, sel1 = (2 + ((lane & 3) >> 1)) * 0x11u;
        const uint32_t boff = static_cast<uint32_t>((4 * min(g, M - 1) + c) * 16);
        float* mine = part + warp * M * a.rows_pad;
        for (int e = lane; e < M * a.rows_pad; e += 32) mine[e] = 0.0f;
        const uint16_t* xs = reinterpret_cast<const uint16_t*>(base + a.off_x);  // [M][xk] bf16: the CTA's units
        if (warp == 0) {
            griddep_wait();  // X belongs to the previous grid until now
            if (lane == 0) {
                const uint32_t row = static_cast<uint32_t>(xk) * 2u;
                mbar_arrive_expect_tx(xfull, row * static_cast<uint32_t>(M));
                for (int m = 0; m < M; ++m)
                    bulk_g2s_plain(smem_addr(xs) + m * row, a.X + static_cast<size_t>(m) * a.K + ua * kUnitK, row, xfull);
            }
            __syncwarp();
        }
        if (lane == 0) mbar_arrive(xreq);
        bool ok = mbar_wait_warp(xfull, 0);
        if (ok)
            for (int p = warp; p < U * M; p += kNrWarps) {
                const int u = p / M, m = p - u * M;
                nv_build_row_compact<LR>(rec(u), so(u), xs + static_cast<size_t>(m) * xk + u * kUnitK, m, a.g, lane);
            }
        named_sync(1, 32 * kNrWarps);
        int k0 = warp;
        for (int s = 0, i = 0, j = 0; ok && s < nstages; ++s) {
            const int slot = s % S;
            if (!mbar_wait_warp(full(slot), (s / S) & 1)) {
                ok = false;
                break;
            }
            const int u0 = seg_tab[j], n = seg_tab[j + 1] - u0;
            const uint32_t pc = static_cast<uint32_t>(nr_pitch(n * 128)), ps = static_cast<uint32_t>(nr_pitch(n * 16));
            const uint32_t st = smem_addr(stage(slot));
            const uint32_t c0 = st + g * pc + 4u * c, s0 = st + a.scale_region + g * ps;
            if (k0 < n) {
                float t0 = 0.0f, t1 = 0.0f;  // rows g, g + 8 of activation row c (c < M)
                for (int k = k0; k < n; k += kNrWarps) {
                    const int u = u0 + k;
                    const uint32_t scode[2] = {c0 + 128u * k, c0 + 8u * pc + 128u * k};
                    const uint32_t sscl[2] = {s0 + 16u * k, s0 + 8u * ps + 16u * k};
                    float acc[4];
                    nv_task<LR>(scode, sscl, smem_addr(rec(u)) + boff, c, sel0, sel1, acc);
                    // column 2c' + i of the mma is activation row m = ... : the live columns are m < M
                    // (one column per row); lane c holds columns 2c and 2c + 1
                    const float* f = so(u);
                    if (2 * c < M) {
                        t0 = fmaf(acc[0], f[2 * c], t0);
                        t1 = fmaf(acc[2], f[2 * c], t1);
                    }
                    if (2 * c + 1 < M) {
                        mine[(2 * c + 1) * a.rows_pad + i * kGroupRows + g] += acc[1] * f[2 * c + 1];
                        mine[(2 * c + 1) * a.rows_pad + i * kGroupRows + g + 8] += acc[3] * f[2 * c + 1];
                    }
                }
                if (2 * c < M) {
                    mine[(2 * c) * a.rows_pad + i * kGroupRows + g] += t0;
                    mine[(2 * c) * a.rows_pad + i * kGroupRows + g + 8] += t1;
                }
            }
            k0 = (k0 - n) & (kNrWarps - 1);
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(slot));
            if (++j == nseg) {
                j = 0;
                ++i;
            }
        }
        if (!ok && lane == 0) record_error(a.err, kErrFullWait);
    }

    __syncthreads();
    if (CL == 1) {
        griddep_wait();  // Y may still be read by the previous grid
        for (int e = threadIdx.x; e < M * nrows; e += kNrThreads) {
            const int m = e / nrows, r = e - m * nrows;
            float v = 0.0f;
            for (int w = 0; w < kNrWarps; ++w) v += part[(w * M + m) * a.rows_pad + r];
            a.Y[static_cast<size_t>(m) * a.N + r0 + r] = v;
        }
        return;
    }
    // this CTA's sum over its warps, in warp 0's slice; then CTA cr writes a share of the rows
    // from the sums of every CTA of the cluster (distributed shared memory, CTA order)
    for (int e = threadIdx.x; e < M * nrows; e += kNrThreads) {
        const int m = e / nrows, r = e - m * nrows;
        float v = 0.0f;
        for (int w = 0; w < kNrWarps; ++w) v += part[(w * M + m) * a.rows_pad + r];
        part[m * a.rows_pad + r] = v;
    }
    cluster_sync();
    griddep_wait();  // Y may still be read by the previous grid
    {
        const int E = M * nrows, e0 = cr * E / CL, e1 = (cr + 1) * E / CL;
        const uint32_t pbase = smem_addr(part);
        for (int e = e0 + static_cast<int>(threadIdx.x); e < e1; e += kNrThreads) {
            const int m = e / nrows, r = e - m * nrows;
            const uint32_t off = 4u * static_cast<uint32_t>(m * a.rows_pad + r);
            float v = 0.0f;
            for (int q = 0; q < CL; ++q) v += ld_dsmem_f32(pbase + off, static_cast<uint32_t>(q));
            a.Y[static_cast<size_t>(m) * a.N + r0 + r] = v;
        }
    }
    cluster_sync();  // no CTA leaves while another still reads its sums
}

// Plan: grid (clusters of CL CTAs splitting K, one CTA per SM, no more clusters than can be
// resident when max_clusters > 0), segments of one CTA's units (whole rows of at most 20 units,
// else segments of at most 8, 6, 4 units), the deepest ring of 8..3 stages (2 as a last resort);
// false when nothing fits.
template <int LR>
bool nr_plan(int64_t N, int Ut, int M, int sms, NrArgs& a, uint32_t& total, int CL = 1, int max_clusters = 0) {
    constexpr int REC = 8 * LR * 16;
    if (CL < 1 || CL > 8 || sms / CL < 1 || Ut < CL) return false;
    const int U = (Ut + CL - 1) / CL;  // the most units of a CTA
    if (U < 1 || M < 1 || 4 * M > LR || (U + 3) / 4 > kNrMaxSeg) return false;
    a.CL = CL;
    const int ncl = max_clusters > 0 ? std::min(sms / CL, max_clusters) : sms / CL;
    a.G = static_cast<int>(std::min<int64_t>(ncl, N));
    const int64_t rows_max = (N + a.G - 1) / a.G;
    a.rows_pad = static_cast<int>((rows_max + kGroupRows - 1) / kGroupRows * kGroupRows);
    a.off_rec = align_up(8u * (2u * kNrMaxStages + 2), 128);
    a.off_so = align_up(a.off_rec + static_cast<uint32_t>(U) * REC, 16);
    a.off_x = align_up(a.off_so + static_cast<uint32_t>(U) * kNrMaxM * 4u, 16);
    a.off_part = align_up(a.off_x + static_cast<uint32_t>(M) * U * kUnitK * 2u, 16);
    a.off_stage = align_up(a.off_part + kNrWarps * static_cast<uint32_t>(M * a.rows_pad) * 4u, 128);
    const int cap[4] = {20, 8, 6, 4};
    for (int s_lo : {3, 2})
        for (int t = 0; t < 4; ++t) {
            a.nseg = (U + cap[t] - 1) / cap[t];
            const int longest = (U + a.nseg - 1) / a.nseg;
            a.scale_region = align_up(static_cast<uint32_t>(kGroupRows * nr_pitch(longest * 128)), 16);
            a.stage_bytes = align_up(a.scale_region + static_cast<uint32_t>(kGroupRows * nr_pitch(longest * 16)), 128);
            for (int S = kNrMaxStages; S >= s_lo; --S) {
                a.S = S;
                total = a.off_stage + static_cast<uint32_t>(S) * a.stage_bytes;
                if (total + 1024u <= kNrSmem) return true;
            }
        }
    return false;
}

// Estimated time (us) of an NVFP4 row-stream plan, fitted like the PN one to both NVFP4 shapes
// at M = 1, 2, 4, 8 with every cluster size forced: ~2.5 us until the first stage is multiplied,
// 0.2 us per further round of operand builds, the longer of the dealt tasks (0.5 us per 16 rows
// x one 256-weight unit) and the weight stream, and 1.5 us for a cluster's final sum. The stream
// takes at least ~0.8 us per stage however small its copies (each stage is 32 of them), and
// runs at 35 GB/s per SM or at the ring's pace when that is slower: the S - 1 stages in flight
// over a ~1.8 us round trip.
inline double nr_cost(const NrArgs& a, int64_t N, int Ut, int M) {
    const int U = (Ut + a.CL - 1) / a.CL;
    const int64_t rows = (N + a.G - 1) / a.G;
    const int64_t groups = (rows + kGroupRows - 1) / kGroupRows;
    const double tasks = static_cast<double>((groups * U + kNrWarps - 1) / kNrWarps);
    const double builds = static_cast<double>((U * M + kNrWarps - 1) / kNrWarps);
    const double rate = std::min(35e3, std::max(1, a.S - 1) * static_cast<double>(a.stage_bytes) / 1.8);  // bytes / us
    const double stream = std::max(static_cast<double>(rows) * U * 144.0 / rate, 0.8 * static_cast<double>(groups * a.nseg));
    return 2.5 + 0.2 * (builds - 1.0) + std::max(0.5 * tasks, stream) + (a.CL > 1 ? 1.5 : 0.0);
}

// Clusters of CL CTAs of the row kernel that can be resident at once (0 when the query fails).
template <int LR>
int nv_rows_resident_clusters(int CL, int ncl, uint32_t total) {
    if (cudaFuncSetAttribute(nv_rows_kernel<LR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kNrSmem)) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(ncl * CL, 1, 1);
    lc.blockDim = dim3(kNrThreads, 1, 1);
    lc.dynamicSmemBytes = total + 1024u;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(CL);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, nv_rows_kernel<LR>, &lc) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

// The cheapest plan over clusters of 1, 2, 4 and 8 CTAs (cl_req > 0: that size only), cached per
// device and shape.
template <int LR>
bool nr_best_plan(int64_t N, int U, int M, int cl_req, NrArgs& a, uint32_t& total) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    using Key = std::tuple<int, int64_t, int, int, int>;
    static std::mutex mu;
    static std::map<Key, std::pair<NrArgs, uint32_t>> cache;
    const Key key{dev, N, U, M, cl_req};
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) {
            a = it->second.first;
            total = it->second.second;
            return true;
        }
    }
    const int sms = device_sm_count();
    bool found = false;
    double best = 0.0;
    for (int CL : {1, 2, 4, 8}) {
        if (cl_req > 0 && CL != cl_req) continue;
        NrArgs q{};
        uint32_t t = 0;
        if (!nr_plan<LR>(N, U, M, sms, q, t, CL)) continue;
        if (CL > 1) {
            const int most = nv_rows_resident_clusters<LR>(CL, q.G, t);
            if (most < 1) continue;
            if (most < q.G && !nr_plan<LR>(N, U, M, sms, q, t, CL, most)) continue;
        }
        const double cost = nr_cost(q, N, U, M);
        if (!found || cost < best) {
            a = q;
            total = t;
            best = cost;
            found = true;
        }
    }
    if (!found) return false;
    std::lock_guard<std::mutex> lock(mu);
    if (cache.size() < 4096) cache.emplace(key, std::make_pair(a, total));
    return true;
}

template <int LR>
cudaError_t launch_nv_rows(const Nvfp4View& w, int64_t N, int64_t K, const uint16_t* X, int M, float* Y, int* err,
                           bool static_weights, int cl_req, cudaStream_t stream) {
    NrArgs a{};
    uint32_t total = 0;
    if (!nr_best_plan<LR>(N, static_cast<int>(K / kUnitK), M, cl_req, a, total)) return cudaErrorNotSupported;
    a.codes = w.codes;
    a.scales = w.scales;
    a.X = X;
    a.Y = Y;
    a.err = err;
    a.g = w.g;
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.M = M;
    a.U = static_cast<int>(K / kUnitK);
    a.flags = static_weights ? kStaticWeights : 0u;
    auto kern = nv_rows_kernel<LR>;
    static std::atomic<bool> opted[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!opted[dev].load(std::memory_order_relaxed)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kNrSmem));
        if (e != cudaSuccess) return e;
        opted[dev].store(true, std::memory_order_relaxed);
    }
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(a.G * a.CL, 1, 1);
    lc.blockDim = dim3(kNrThreads, 1, 1);
    lc.dynamicSmemBytes = total + 1024u;
    lc.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(a.CL);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 2;
    return cudaLaunchKernelEx(&lc, kern, a);
}

template <int NT>
cudaError_t launch_nt(const CUtensorMap (&maps)[4], float g, const uint16_t* X, float* Y, int* err, int64_t N,
                      int64_t K, int M, int U, const int (&req)[3], bool static_weights, cudaStream_t stream) {
    KArgs<NvMma<NT>> ka{};
    for (int i = 0; i < 4; ++i) ka.map[i] = maps[i];
    ka.e.g = g;
    ka.c.X = X;
    ka.c.Y = Y;
    ka.c.err = err;
    ka.c.N = static_cast<int>(N);
    ka.c.K = static_cast<int>(K);
    ka.c.M = M;
    return cl_launch<NvMma<NT>>(ka, N, U, req, static_weights, stream);
}

}  // namespace

cudaError_t launch_nvfp4_gemv_mma(const Nvfp4View& w, int64_t N, int64_t K, const uint16_t* X, int M, float* Y,
                                  int* err, int c_req, int s_req, bool static_weights, cudaStream_t stream) {
    if (N == 0) return cudaSuccess;
    if (K % kUnitK != 0 || M < 1 || M > 16) return cudaErrorNotSupported;
    if (N > INT32_MAX - 64 || K > INT32_MAX) return cudaErrorNotSupported;
    if (reinterpret_cast<uintptr_t>(w.codes) % 16 != 0 || reinterpret_cast<uintptr_t>(w.scales) % 16 != 0 ||
        reinterpret_cast<uintptr_t>(X) % 16 != 0)
        return cudaErrorNotSupported;
    CUtensorMap maps[4];
    if (!encode_u32_map(&maps[0], w.codes, N, K / 8, kCodeRow / 4, kPieceRows, true) ||
        !encode_u32_map(&maps[1], w.scales, N, K / 64, kScaleRow / 4, kPieceRows, false) ||
        !encode_u32_map(&maps[2], w.codes, N, K / 8, kCodeRow / 4, kStageRows, true) ||
        !encode_u32_map(&maps[3], w.scales, N, K / 64, kScaleRow / 4, kStageRows, false))
        return cudaErrorNotSupported;
    // PNQ_NV_CFG = "CTAs per cluster, stages, CTAs per SM (strip pipeline), CTAs per cluster splitting K
    // (row stream; 0: cheapest)", read once
    static int env[4];
    static std::once_flag once;
    std::call_once(once, [] { env_cluster_config("PNQ_NV_CFG", env); });
    const int req[3] = {c_req > 0 ? c_req : env[0], s_req > 0 ? s_req : env[1], env[2]};
    const int U = static_cast<int>(K / kUnitK);
    // the row stream when a CTA's units' B records and x fit beside the ring (M <= 8: one column
    // per activation row, so one n8 tile)
    if (M <= 8 && c_req <= 0 && env[0] == 0 && env[1] == 0) {
        const int cl = env[3];
        const cudaError_t e = (M == 1)   ? launch_nv_rows<4>(w, N, K, X, M, Y, err, static_weights, cl, stream)
                              : (M == 2) ? launch_nv_rows<8>(w, N, K, X, M, Y, err, static_weights, cl, stream)
                              : (M == 3) ? launch_nv_rows<12>(w, N, K, X, M, Y, err, static_weights, cl, stream)
                              : (M == 4) ? launch_nv_rows<16>(w, N, K, X, M, Y, err, static_weights, cl, stream)
                                         : launch_nv_rows<32>(w, N, K, X, M, Y, err, static_weights, cl, stream);
        if (e != cudaErrorNotSupported) return e;
    }
    if (M <= 8) return launch_nt<1>(maps, w.g, X, Y, err, N, K, M, U, req, static_weights, stream);
    return launch_nt<2>(maps, w.g, X, Y, err, N, K, M, U, req, static_weights, stream);
}

}  // namespace pnq
