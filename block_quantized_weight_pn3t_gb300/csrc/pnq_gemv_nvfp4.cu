// pnq_gemv_nvfp4.cu -- NVFP4 (W4A16) GEMV on the tensor cores with mma.sync, sm_103a (fast path).
//
// Computes Y[m][n] = sum_k w[n][k] x[m][k] for 1 <= M <= 16 with w = e2m1(code) * e4m3(scale) * g
// ("Quantisation and profiles", NVFP4; tensor-formats page, NVFP4 / E2M1 / E4M3FN): codes two per
// byte, low nibble = even k, one E4M3FN scale per 16 weights along K, one fp32 global multiplier;
// x is bf16. The weights are decoded in registers just before the multiply. The pipeline (cluster
// work split, weight stream, operand builders, on-chip reduction) is pnq_cluster.cuh; this file is
// the NVFP4 format policy.
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
    static int env[3];  // PNQ_NV_CFG = "CTAs per cluster, stages, CTAs per SM", read once
    static std::once_flag once;
    std::call_once(once, [] { env_cluster_config("PNQ_NV_CFG", env); });
    const int req[3] = {c_req > 0 ? c_req : env[0], s_req > 0 ? s_req : env[1], env[2]};
    const int U = static_cast<int>(K / kUnitK);
    if (M <= 8) return launch_nt<1>(maps, w.g, X, Y, err, N, K, M, U, req, static_weights, stream);
    return launch_nt<2>(maps, w.g, X, Y, err, N, K, M, U, req, static_weights, stream);
}

}  // namespace pnq
