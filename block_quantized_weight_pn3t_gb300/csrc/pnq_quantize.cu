// pnq_quantize.cu -- the PN reference quantizer ("PN weight format", section Reference quantizer)
// on the GPU, bit for bit the CPU reference's choice of d and codes.
//
// Per block of BLK weights: amax, max and min; amax == 0 gives the canonical zero block (d = +0,
// every code z). Otherwise sigma = +1 when |min| > max, else -1, and for the 36 multipliers
// m = 0.50, 0.52, .., 1.20 the candidate scale is s = fp16(sigma * m * amax / z) (skipped when
// it is zero or not finite), the codes n = clamp(rint(w / s) + z, 0, 2z - 1) and the error
// sum over the block of (w - s (n - z))^2; the smallest error wins, a tie going to the larger m,
// and d = s. Readings where the page is silent: m = (50 + 2i) / 100 in double, the fp16 rounding
// a single round-to-nearest-even step from double, every other step one IEEE double operation in
// the order written (no fused multiply-add), the error summed in element order, and a block whose
// every candidate is skipped written as the canonical zero block.
//
// One warp per block: lane i scores multiplier i (lanes 0..3 also score 32..35), each summing its
// block in element order so the result does not depend on the warp's layout; the winner is reduced
// across the warp, its codes are packed into the eight words (element e in word e / CPW at shift
// BITS * (t >> 1) + 16 * (t & 1), t = e mod CPW) and the 34-byte block is written with 16-bit
// stores (a block of a row starts on any even byte).
#include "pnq_device.cuh"
#include "pnq_internal.h"

#include <cuda_fp16.h>

#include <algorithm>

namespace pnq {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kCandidates = 36;

// binary16 bits of a double, rounded once to nearest even; overflow gives infinity. Written from
// the binary64 and binary16 encodings: keep 11 significant bits of the value (fewer below 2^-14,
// where the binary16 spacing is 2^-24) and round the rest half to even.
__device__ __forceinline__ uint16_t f64_to_f16_rne(double x) {
    const unsigned long long b = static_cast<unsigned long long>(__double_as_longlong(x));
    const uint16_t sign = static_cast<uint16_t>((b >> 48) & 0x8000u);
    const int e = static_cast<int>((b >> 52) & 0x7FF);
    const unsigned long long f = b & 0xFFFFFFFFFFFFFull;
    if (e == 0x7FF) return sign | (f ? 0x7E00u : 0x7C00u);
    if (e == 0) return sign;  // binary64 zero or subnormal: far below half the smallest binary16
    const int E = e - 1023;   // value = 1.f * 2^E
    // significand with the implicit bit, 53 bits; binary16 keeps bits down to 2^max(E - 10, -24)
    const unsigned long long sig = f | (1ull << 52);
    const int keep_lsb = (E >= -14) ? E - 10 : -24;  // exponent of the last kept bit
    const int drop = 52 - (E - keep_lsb);            // low bits of sig below that bit
    if (drop > 53) return sign;                      // below 2^-25: rounds to zero
    unsigned long long q = sig >> drop;
    const unsigned long long rem = sig & ((1ull << drop) - 1ull), half = 1ull << (drop - 1);
    if (rem > half || (rem == half && (q & 1ull))) ++q;  // q counts units of 2^keep_lsb
    // value = q * 2^keep_lsb; encode (q may have carried into a new binade)
    if (keep_lsb == -24) {
        if (q < 1024ull) return sign | static_cast<uint16_t>(q);  // subnormal
        return sign | static_cast<uint16_t>((1u << 10) | (q - 1024ull));  // first normal binade (q == 1024)
    }
    int E2 = E;
    if (q == (1ull << 11)) {
        q >>= 1;
        ++E2;
    }
    if (E2 > 15) return sign | 0x7C00u;
    return sign | static_cast<uint16_t>(((E2 + 15) << 10) | static_cast<int>(q & 0x3FFull));
}

template <int TYPE>
__global__ void __launch_bounds__(kThreads) pn_quantize_kernel(const float* __restrict__ w, int64_t nblocks,
                                                                 int64_t blocks_per_row, uint8_t* __restrict__ out,
                                                                 int32_t* __restrict__ status) {
    using F = PnFmt<TYPE>;
    constexpr int BLK = F::BLK, Z = F::Z;
    __shared__ float sw[kWarps][BLK];
    __shared__ int scode[kWarps][BLK];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarps;
    for (int64_t blk = static_cast<int64_t>(blockIdx.x) * kWarps + warp; blk < nblocks; blk += stride) {
        float* x = sw[warp];
        bool finite = true;
        float amax = 0.0f, mx = -INFINITY, mn = INFINITY;
        for (int k = lane; k < BLK; k += 32) {
            const float v = __ldg(w + blk * BLK + k);
            x[k] = v;
            finite &= isfinite(v);
            amax = fmaxf(amax, fabsf(v));
            mx = fmaxf(mx, v);
            mn = fminf(mn, v);
        }
        __syncwarp();
        if (!__all_sync(0xffffffffu, finite)) {
            if (lane == 0) status[blk / blocks_per_row] = 1;
            continue;
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, d));
        }
        uint16_t dbits = 0;
        double s = 0.0;
        bool any = false;
        if (amax != 0.0f) {
            const double sigma = (fabs(static_cast<double>(mn)) > static_cast<double>(mx)) ? 1.0 : -1.0;
            // score candidates lane and (lanes 0..3) 32 + lane; keep the lane's better one
            double best = 0.0;
            int best_i = -1;
            for (int i = lane; i < kCandidates; i += 32) {
                const double m = __ddiv_rn(static_cast<double>(50 + 2 * i), 100.0);
                const uint16_t sb = f64_to_f16_rne(
                    __ddiv_rn(__dmul_rn(__dmul_rn(sigma, m), static_cast<double>(amax)), static_cast<double>(Z)));
                const double sv = static_cast<double>(__half2float(__ushort_as_half(sb)));
                if (sv == 0.0 || !isfinite(sv)) continue;
                double err = 0.0;
                for (int k = 0; k < BLK; ++k) {
                    const double wd = static_cast<double>(x[k]);
                    double q = __dadd_rn(rint(__ddiv_rn(wd, sv)), static_cast<double>(Z));
                    q = fmin(fmax(q, 0.0), static_cast<double>(2 * Z - 1));
                    const double diff = __dsub_rn(wd, __dmul_rn(sv, __dsub_rn(q, static_cast<double>(Z))));
                    err = __dadd_rn(err, __dmul_rn(diff, diff));
                }
                if (best_i < 0 || err <= best) {  // i ascends: a tie goes to the larger m
                    best = err;
                    best_i = i;
                }
            }
            // across the warp: smallest error, then the largest index
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) {
                const double ob = __shfl_xor_sync(0xffffffffu, best, d);
                const int oi = __shfl_xor_sync(0xffffffffu, best_i, d);
                if (oi >= 0 && (best_i < 0 || ob < best || (ob == best && oi > best_i))) {
                    best = ob;
                    best_i = oi;
                }
            }
            if (best_i >= 0) {
                any = true;
                const double m = __ddiv_rn(static_cast<double>(50 + 2 * best_i), 100.0);
                dbits = f64_to_f16_rne(
                    __ddiv_rn(__dmul_rn(__dmul_rn(sigma, m), static_cast<double>(amax)), static_cast<double>(Z)));
                s = static_cast<double>(__half2float(__ushort_as_half(dbits)));
            }
        }
        for (int k = lane; k < BLK; k += 32) {
            int n = Z;
            if (any) {
                double q = __dadd_rn(rint(__ddiv_rn(static_cast<double>(x[k]), s)), static_cast<double>(Z));
                q = fmin(fmax(q, 0.0), static_cast<double>(2 * Z - 1));
                n = static_cast<int>(q);
            }
            scode[warp][k] = n;
        }
        __syncwarp();
        // lane i < 8 packs word i; lanes write the block as 17 halves: d, then the words' halves
        uint32_t word = 0;
        if (lane < 8)
            for (int t = 0; t < F::CPW; ++t)
                word |= static_cast<uint32_t>(scode[warp][lane * F::CPW + t]) << (F::BITS * (t >> 1) + 16 * (t & 1));
        const uint32_t wsrc = __shfl_sync(0xffffffffu, word, (lane - 1) >> 1 & 7);
        uint16_t* dst = reinterpret_cast<uint16_t*>(out + blk * kBlockBytes);
        if (lane == 0) dst[0] = dbits;
        if (lane >= 1 && lane <= 16) dst[lane] = static_cast<uint16_t>(((lane - 1) & 1) ? (wsrc >> 16) : (wsrc & 0xFFFFu));
        __syncwarp();
    }
}

// ---- NVFP4 clip search (TandemLLM "Quantisation and profiles", section "The clip search") ----
// Per group of 16 weights of a row, the multipliers 1.00, 0.95, 0.90, 0.85, 0.80 of the base scale
// amax / (6 g) are tried and the one with the least sum_k act_ms[k] (w[k] - dq[k])^2 kept, the
// same choice as the CPU reference bit for bit. Readings where the page is silent: the scale
// ((mu * amax) / 6) / g is rounded to the nearest E4M3FN value (ties to the even word,
// saturating at 448); a weight takes the nearest E2M1 magnitude of |w| / (scale * g) (ties to the
// even word, saturating at 6) with the sign of w; a zero scale gives zero words; the error is
// summed in k order; a tie keeps the earlier multiplier; every step one IEEE double operation.
// One thread per group (16 weights, five candidates; nearest values by scanning the 127 finite
// positive E4M3FN words and the 8 E2M1 magnitudes).

__device__ __forceinline__ double e4m3_value(int c) {  // c in 0 .. 0x7E: exact in double
    const int e = (c >> 3) & 15, m = c & 7;
    return e == 0 ? static_cast<double>(m) * 0x1p-9 : (1.0 + m * 0.125) * exp2(static_cast<double>(e - 7));
}

__device__ __forceinline__ double e2m1_value(int c) {  // c in 0 .. 7
    const int e = (c >> 1) & 3, m = c & 1;
    return e == 0 ? 0.5 * m : (1.0 + 0.5 * m) * exp2(static_cast<double>(e - 1));
}

__global__ void __launch_bounds__(kThreads) nvfp4_clip_kernel(const float* __restrict__ w,
                                                               const float* __restrict__ act_ms, double gd,
                                                               int64_t n_rows, int64_t K, uint8_t* __restrict__ codes,
                                                               uint8_t* __restrict__ scales,
                                                               int32_t* __restrict__ status) {
    const double kMu[5] = {1.00, 0.95, 0.90, 0.85, 0.80};
    const int64_t gpr = K / 16, total = n_rows * gpr;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total; t += stride) {
        const int64_t r = t / gpr, grp = t - r * gpr;
        float x[16], a[16];
        double amax = 0.0;
        bool finite = true;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            x[k] = __ldg(w + r * K + grp * 16 + k);
            a[k] = __ldg(act_ms + grp * 16 + k);
            finite &= isfinite(x[k]);
            amax = fmax(amax, fabs(static_cast<double>(x[k])));
        }
        if (!finite) {
            status[r] = 1;
            continue;
        }
        double best = 0.0;
        int best_sc = 0;
        uint8_t best_c[16];
        for (int i = 0; i < 5; ++i) {
            const double tgt = __ddiv_rn(__ddiv_rn(__dmul_rn(kMu[i], amax), 6.0), gd);
            int sc = 0;
            double bd = INFINITY;
            for (int c = 0; c <= 0x7E; ++c) {
                const double d = fabs(__dsub_rn(e4m3_value(c), tgt));
                if (d < bd || (d == bd && (c & 1) == 0)) {
                    bd = d;
                    sc = c;
                }
            }
            const double sv = e4m3_value(sc), step = __dmul_rn(sv, gd);
            uint8_t cw[16];
            double err = 0.0;
            for (int k = 0; k < 16; ++k) {
                const int sign = (x[k] < 0.0f || (x[k] == 0.0f && signbit(x[k]))) ? 8 : 0;
                int mag = 0;
                if (sv != 0.0) {
                    const double v = __ddiv_rn(fabs(static_cast<double>(x[k])), step);
                    double md = INFINITY;
                    for (int c = 0; c <= 7; ++c) {
                        const double d = fabs(__dsub_rn(e2m1_value(c), v));
                        if (d < md || (d == md && (c & 1) == 0)) {
                            md = d;
                            mag = c;
                        }
                    }
                }
                cw[k] = static_cast<uint8_t>(sign | mag);
                const double e2 = sign ? -e2m1_value(mag) : e2m1_value(mag);
                const double dq = __dmul_rn(__dmul_rn(e2, sv), gd);
                const double diff = __dsub_rn(static_cast<double>(x[k]), dq);
                err = __dadd_rn(err, __dmul_rn(static_cast<double>(a[k]), __dmul_rn(diff, diff)));
            }
            if (i == 0 || err < best) {
                best = err;
                best_sc = sc;
#pragma unroll
                for (int k = 0; k < 16; ++k) best_c[k] = cw[k];
            }
        }
        scales[r * gpr + grp] = static_cast<uint8_t>(best_sc);
#pragma unroll
        for (int k = 0; k < 16; k += 2)
            codes[r * (K / 2) + grp * 8 + k / 2] = static_cast<uint8_t>(best_c[k] | (best_c[k + 1] << 4));
    }
}

int quant_grid(int64_t nblocks) {
    const int64_t blocks = (nblocks + kWarps - 1) / kWarps;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
    return static_cast<int>(std::max<int64_t>(1, std::min(blocks, cap)));
}

}  // namespace

cudaError_t launch_nvfp4_clip(const float* w, const float* act_ms, float g, int64_t n_rows, int64_t K, uint8_t* codes,
                              uint8_t* scales, int32_t* status, cudaStream_t stream) {
    if (n_rows == 0) return cudaSuccess;
    const cudaError_t e = cudaMemsetAsync(status, 0, static_cast<size_t>(n_rows) * sizeof(int32_t), stream);
    if (e != cudaSuccess) return e;
    const int64_t groups = n_rows * (K / 16);
    const int grid = static_cast<int>(
        std::max<int64_t>(1, std::min<int64_t>((groups + kThreads - 1) / kThreads, int64_t(device_sm_count()) * 8)));
    nvfp4_clip_kernel<<<grid, kThreads, 0, stream>>>(w, act_ms, static_cast<double>(g), n_rows, K, codes, scales,
                                                     status);
    return cudaGetLastError();
}

cudaError_t launch_pn_quantize(int type, const float* w, int64_t n_rows, int64_t K, uint8_t* out, int32_t* status,
                               cudaStream_t stream) {
    if (n_rows == 0) return cudaSuccess;
    const cudaError_t e = cudaMemsetAsync(status, 0, static_cast<size_t>(n_rows) * sizeof(int32_t), stream);
    if (e != cudaSuccess) return e;
    const int blk = (type == kTypePn3t) ? PnFmt<kTypePn3t>::BLK : PnFmt<kTypePn4t>::BLK;
    const int64_t bpr = K / blk, nblocks = n_rows * bpr;
    if (type == kTypePn3t)
        pn_quantize_kernel<kTypePn3t><<<quant_grid(nblocks), kThreads, 0, stream>>>(w, nblocks, bpr, out, status);
    else
        pn_quantize_kernel<kTypePn4t><<<quant_grid(nblocks), kThreads, 0, stream>>>(w, nblocks, bpr, out, status);
    return cudaGetLastError();
}

}  // namespace pnq
