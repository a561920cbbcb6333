// pnq_grouped.cu -- the grouped signed-integer weight formats of NInfer "tensor-formats.md"
// (sections 4 to 7): Q4G64_F16S, Q5G64_F16S, Q6G64_F16S and W8G32_F16S. Dequantize, validate,
// GEMV on the CUDA cores and the canonical encoder MAXABS_F16_RECIP_RNE_V1.
//
// A row of K weights (K % 8 == 0) holds one two's-complement code per weight and one binary16
// scale per group of G = 64 (32 for W8) along K, the last group possibly partial. The represented
// weight is binary32(s32 * binary32(q)) (section 6.2): a binary16 scale has 11 significant bits
// and a code at most 8, so the fp32 product is exact and a dequantize is bit-exact by construction.
//
// Plane layout (the pages leave it to a layout registry; this is the library's own): the low 4
// bits of each logical word in a nibble plane lo[N][K/2] (even k in the low nibble), the bits above
// in a plane hi (Q5: hi[N][K/8], bit k % 8 of byte k / 8; Q6: hi[N][K/4], bits 2 (k % 4) and up
// of byte k / 4); W8 keeps its byte per weight in lo[N][K] and has no hi plane; scales
// sc[N][ceil(K / G)]. The unit of work is an octet of 8 consecutive weights: 4 bytes of the nibble
// plane (8 for W8), one byte (Q5) or two (Q6) of the high plane, and one scale (G is a multiple
// of 8, so an octet never straddles a group).
#include "pnq_device.cuh"
#include "pnq_internal.h"

#include <cuda_fp16.h>

#include <algorithm>

namespace pnq {
namespace {

constexpr int kThreads = 256;

int grid_for(int64_t items) {
    const int64_t blocks = (items + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
    return static_cast<int>(std::max<int64_t>(1, std::min(blocks, cap)));
}

// Per-scheme constants: code width, group, code interval (section 5).
template <int BITS>
struct Grp {
    static constexpr int G = (BITS == 8) ? 32 : 64;
    static constexpr int QMAX = (BITS == 8) ? 127 : (1 << (BITS - 1)) - 1;
    static constexpr int QMIN = (BITS == 8) ? -127 : -(1 << (BITS - 1));
};

// The 8 signed codes of octet o of a row (lo / hi: the row's planes).
template <int BITS>
__device__ __forceinline__ void octet_codes(const uint8_t* __restrict__ lo, const uint8_t* __restrict__ hi,
                                            int64_t o, int (&q)[8]) {
    if constexpr (BITS == 8) {
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(lo) + o);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            q[j] = static_cast<int8_t>((v.x >> (8 * j)) & 0xFFu);
            q[4 + j] = static_cast<int8_t>((v.y >> (8 * j)) & 0xFFu);
        }
    } else {
        const uint32_t l = __ldg(reinterpret_cast<const uint32_t*>(lo) + o);
        uint32_t h = 0;
        if constexpr (BITS == 5) h = __ldg(hi + o);
        if constexpr (BITS == 6) h = __ldg(reinterpret_cast<const uint16_t*>(hi) + o);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint32_t u = (l >> (4 * j)) & 15u;
            if constexpr (BITS == 5) u |= ((h >> j) & 1u) << 4;
            if constexpr (BITS == 6) u |= ((h >> (2 * j)) & 3u) << 4;
            // two's complement of BITS bits (section 5): sign-extend from bit BITS - 1
            q[j] = static_cast<int>(u << (32 - BITS)) >> (32 - BITS);
        }
    }
}

// One thread per octet: 8 exact products, written as two 16-byte stores.
template <int BITS>
__global__ void __launch_bounds__(kThreads) grouped_dequant_kernel(const uint8_t* __restrict__ lo,
                                                                     const uint8_t* __restrict__ hi,
                                                                     const uint16_t* __restrict__ sc, int64_t n_rows,
                                                                     int64_t K, float* __restrict__ out) {
    using P = Grp<BITS>;
    const int64_t opr = K / 8, ns = (K + P::G - 1) / P::G, total = n_rows * opr;
    const int64_t lb = (BITS == 8) ? K : K / 2, hb = (BITS == 5) ? K / 8 : (BITS == 6) ? K / 4 : 0;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t r = i / opr, o = i - r * opr;
        int q[8];
        octet_codes<BITS>(lo + r * lb, hi + r * hb, o, q);
        const float s = __half2float(__ushort_as_half(__ldg(sc + r * ns + (o * 8) / P::G)));
        float4* dst = reinterpret_cast<float4*>(out + r * K + o * 8);
        dst[0] = make_float4(__fmul_rn(s, static_cast<float>(q[0])), __fmul_rn(s, static_cast<float>(q[1])),
                             __fmul_rn(s, static_cast<float>(q[2])), __fmul_rn(s, static_cast<float>(q[3])));
        dst[1] = make_float4(__fmul_rn(s, static_cast<float>(q[4])), __fmul_rn(s, static_cast<float>(q[5])),
                             __fmul_rn(s, static_cast<float>(q[6])), __fmul_rn(s, static_cast<float>(q[7])));
    }
}

// One warp per row: a scale must be +0 or finite positive; a +0 scale covers only zero codes;
// W8 never holds the word 0x80 (section 6).
template <int BITS>
__global__ void __launch_bounds__(kThreads) grouped_validate_kernel(const uint8_t* __restrict__ lo,
                                                                      const uint8_t* __restrict__ hi,
                                                                      const uint16_t* __restrict__ sc, int64_t n_rows,
                                                                      int64_t K, int32_t* __restrict__ flags) {
    using P = Grp<BITS>;
    const int lane = threadIdx.x & 31;
    const int64_t opr = K / 8, ns = (K + P::G - 1) / P::G;
    const int64_t lb = (BITS == 8) ? K : K / 2, hb = (BITS == 5) ? K / 8 : (BITS == 6) ? K / 4 : 0;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t r = warp0; r < n_rows; r += nwarps) {
        bool bad = false;
        for (int64_t o = lane; o < opr; o += 32) {
            const uint32_t s = __ldg(sc + r * ns + (o * 8) / P::G);
            bad |= (s & 0x8000u) != 0 || (s & 0x7C00u) == 0x7C00u;
            int q[8];
            octet_codes<BITS>(lo + r * lb, hi + r * hb, o, q);
            bool nz = false, m128 = false;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                nz |= q[j] != 0;
                m128 |= q[j] == -128;
            }
            bad |= (s == 0u && nz) || (BITS == 8 && m128);
        }
        bad = __any_sync(0xffffffffu, bad);
        if (lane == 0) flags[r] = bad ? 1 : 0;
    }
}

// GEMV on the CUDA cores, one warp per row; lane l takes octets l, l + 32, ..; per octet the
// 8 products q * x are summed in fp32 and scaled by the octet's scale into the lane's sum.
constexpr int kMaxM = 16;

template <int BITS>
__global__ void __launch_bounds__(kThreads) grouped_gemv_kernel(const uint8_t* __restrict__ lo,
                                                                  const uint8_t* __restrict__ hi,
                                                                  const uint16_t* __restrict__ sc, int64_t N, int64_t K,
                                                                  const float* __restrict__ X, int M,
                                                                  float* __restrict__ Y) {
    using P = Grp<BITS>;
    const int lane = threadIdx.x & 31;
    const int64_t opr = K / 8, ns = (K + P::G - 1) / P::G;
    const int64_t lb = (BITS == 8) ? K : K / 2, hb = (BITS == 5) ? K / 8 : (BITS == 6) ? K / 4 : 0;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t r = warp0; r < N; r += nwarps) {
        float acc[kMaxM];
#pragma unroll
        for (int m = 0; m < kMaxM; ++m) acc[m] = 0.0f;
        for (int64_t o = lane; o < opr; o += 32) {
            int q[8];
            octet_codes<BITS>(lo + r * lb, hi + r * hb, o, q);
            const float s = __half2float(__ushort_as_half(__ldg(sc + r * ns + (o * 8) / P::G)));
#pragma unroll
            for (int m = 0; m < kMaxM; ++m) {
                if (m < M) {
                    const float4* xp = reinterpret_cast<const float4*>(X + m * K + o * 8);
                    const float4 a = __ldg(xp), b = __ldg(xp + 1);
                    float t = static_cast<float>(q[0]) * a.x;
                    t = fmaf(static_cast<float>(q[1]), a.y, t);
                    t = fmaf(static_cast<float>(q[2]), a.z, t);
                    t = fmaf(static_cast<float>(q[3]), a.w, t);
                    t = fmaf(static_cast<float>(q[4]), b.x, t);
                    t = fmaf(static_cast<float>(q[5]), b.y, t);
                    t = fmaf(static_cast<float>(q[6]), b.z, t);
                    t = fmaf(static_cast<float>(q[7]), b.w, t);
                    acc[m] = fmaf(s, t, acc[m]);
                }
            }
        }
#pragma unroll
        for (int m = 0; m < kMaxM; ++m) {
            if (m < M) {
                float v = acc[m];
#pragma unroll
                for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
                if (lane == 0) Y[m * N + r] = v;
            }
        }
    }
}

// Canonical encoder MAXABS_F16_RECIP_RNE_V1 (section 7), one warp per group; lane l holds the
// weights k0 + l * EPL .. + EPL - 1 of the group (EPL = G / 32). Every step is one IEEE operation
// rounded to nearest even, in the page's order: amax; raw = amax / qmax; scale16 = binary16(raw)
// (+0 -> 0x0001, infinity -> the row fails); inv = 1 / scale32; code = clamp(rint(x * inv)).
// A non-finite weight fails the row too; a failed row's planes are left unspecified.
template <int BITS>
__global__ void __launch_bounds__(kThreads) grouped_quantize_kernel(const float* __restrict__ w, int64_t n_rows,
                                                                      int64_t K, uint8_t* __restrict__ lo,
                                                                      uint8_t* __restrict__ hi,
                                                                      uint16_t* __restrict__ sc,
                                                                      int32_t* __restrict__ status) {
    using P = Grp<BITS>;
    constexpr int EPL = P::G / 32;
    const int lane = threadIdx.x & 31;
    const int64_t ns = (K + P::G - 1) / P::G, total = n_rows * ns;
    const int64_t lb = (BITS == 8) ? K : K / 2, hb = (BITS == 5) ? K / 8 : (BITS == 6) ? K / 4 : 0;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t t = warp0; t < total; t += nwarps) {
        const int64_t r = t / ns, g = t - r * ns;
        const int64_t k = g * P::G + lane * EPL;  // the lane's first weight
        const bool live = k < K;                 // K % 8 == 0: a lane's EPL weights are all in or all out
        float x[EPL];
        uint32_t mx = 0;
        bool finite = true;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            x[e] = live ? __ldg(w + r * K + k + e) : 0.0f;
            const uint32_t a = __float_as_uint(x[e]) & 0x7FFFFFFFu;
            finite &= a < 0x7F800000u;
            mx = max(mx, a);  // non-negative floats order like their bits
        }
        mx = __reduce_max_sync(0xffffffffu, mx);
        if (!__all_sync(0xffffffffu, finite)) {
            if (lane == 0) status[r] = 1;
            continue;
        }
        const float amax = __uint_as_float(mx);
        uint16_t s16 = 0;
        float inv = 0.0f;
        if (amax != 0.0f) {
            const float raw = __fdiv_rn(amax, static_cast<float>(P::QMAX));
            s16 = __half_as_ushort(__float2half_rn(raw));
            if (s16 == 0) s16 = 1;  // 2^-24 rescue
            if ((s16 & 0x7C00u) == 0x7C00u) {
                if (lane == 0) status[r] = 1;
                continue;
            }
            inv = __fdiv_rn(1.0f, __half2float(__ushort_as_half(s16)));
        }
        uint32_t u[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            float qf = (amax == 0.0f) ? 0.0f : rintf(__fmul_rn(x[e], inv));
            qf = fminf(fmaxf(qf, static_cast<float>(P::QMIN)), static_cast<float>(P::QMAX));
            u[e] = static_cast<uint32_t>(static_cast<int>(qf)) & ((1u << BITS) - 1u);
        }
        if (lane == 0) sc[r * ns + g] = s16;
        if constexpr (BITS == 8) {
            if (live) lo[r * lb + k] = static_cast<uint8_t>(u[0]);
        } else {
            if (live) lo[r * lb + k / 2] = static_cast<uint8_t>((u[0] & 15u) | ((u[1] & 15u) << 4));
            if constexpr (BITS == 5) {
                // 8 weights (4 lanes) per byte: bit j of the byte is weight 8b + j
                uint32_t bits = ((u[0] >> 4) & 1u) | (((u[1] >> 4) & 1u) << 1);
                bits <<= 2 * (lane & 3);
                bits |= __shfl_xor_sync(0xffffffffu, bits, 1);
                bits |= __shfl_xor_sync(0xffffffffu, bits, 2);
                if (live && (lane & 3) == 0) hi[r * hb + k / 8] = static_cast<uint8_t>(bits);
            } else if constexpr (BITS == 6) {
                // 4 weights (2 lanes) per byte: bits 2j, 2j + 1 of the byte are weight 4b + j
                uint32_t bits = ((u[0] >> 4) & 3u) | (((u[1] >> 4) & 3u) << 2);
                bits <<= 4 * (lane & 1);
                bits |= __shfl_xor_sync(0xffffffffu, bits, 1);
                if (live && (lane & 1) == 0) hi[r * hb + k / 4] = static_cast<uint8_t>(bits);
            }
        }
    }
}

int bits_of(int type) {
    switch (type) {
        case kTypeQ4G64: return 4;
        case kTypeQ5G64: return 5;
        case kTypeQ6G64: return 6;
        case kTypeW8G32: return 8;
        default: return 0;
    }
}

template <template <int> class Launch, typename... A>
cudaError_t by_bits(int type, A&&... args) {
    switch (bits_of(type)) {
        case 4: return Launch<4>::run(args...);
        case 5: return Launch<5>::run(args...);
        case 6: return Launch<6>::run(args...);
        case 8: return Launch<8>::run(args...);
        default: return cudaErrorInvalidValue;
    }
}

template <int BITS>
struct DequantL {
    static cudaError_t run(const GroupedView& v, int64_t n_rows, int64_t K, float* out, cudaStream_t st) {
        grouped_dequant_kernel<BITS><<<grid_for(n_rows * (K / 8)), kThreads, 0, st>>>(v.lo, v.hi, v.scales, n_rows,
                                                                                       K, out);
        return cudaGetLastError();
    }
};

template <int BITS>
struct ValidateL {
    static cudaError_t run(const GroupedView& v, int64_t n_rows, int64_t K, int32_t* flags, cudaStream_t st) {
        grouped_validate_kernel<BITS><<<grid_for(n_rows * 32), kThreads, 0, st>>>(v.lo, v.hi, v.scales, n_rows, K,
                                                                                   flags);
        return cudaGetLastError();
    }
};

template <int BITS>
struct GemvL {
    static cudaError_t run(const GroupedView& v, int64_t N, int64_t K, const float* X, int M, float* Y,
                           cudaStream_t st) {
        grouped_gemv_kernel<BITS><<<grid_for(N * 32), kThreads, 0, st>>>(v.lo, v.hi, v.scales, N, K, X, M, Y);
        return cudaGetLastError();
    }
};

template <int BITS>
struct QuantL {
    static cudaError_t run(const float* w, int64_t n_rows, int64_t K, const GroupedOut& o, int32_t* status,
                           cudaStream_t st) {
        const int64_t groups = n_rows * ((K + Grp<BITS>::G - 1) / Grp<BITS>::G);
        grouped_quantize_kernel<BITS><<<grid_for(groups * 32), kThreads, 0, st>>>(w, n_rows, K, o.lo, o.hi, o.scales,
                                                                                   status);
        return cudaGetLastError();
    }
};

}  // namespace

cudaError_t launch_grouped_dequant(int type, const GroupedView& v, int64_t n_rows, int64_t K, float* out,
                                   cudaStream_t stream) {
    if (n_rows == 0) return cudaSuccess;
    return by_bits<DequantL>(type, v, n_rows, K, out, stream);
}

cudaError_t launch_grouped_validate(int type, const GroupedView& v, int64_t n_rows, int64_t K, int32_t* flags,
                                    cudaStream_t stream) {
    if (n_rows == 0) return cudaSuccess;
    return by_bits<ValidateL>(type, v, n_rows, K, flags, stream);
}

cudaError_t launch_grouped_gemv(int type, const GroupedView& v, int64_t N, int64_t K, const float* X, int M,
                                float* Y, cudaStream_t stream) {
    if (N == 0) return cudaSuccess;
    return by_bits<GemvL>(type, v, N, K, X, M, Y, stream);
}

cudaError_t launch_grouped_quantize(int type, const float* w, int64_t n_rows, int64_t K, const GroupedOut& out,
                                    int32_t* status, cudaStream_t stream) {
    if (n_rows == 0) return cudaSuccess;
    const cudaError_t e = cudaMemsetAsync(status, 0, static_cast<size_t>(n_rows) * sizeof(int32_t), stream);
    if (e != cudaSuccess) return e;
    return by_bits<QuantL>(type, w, n_rows, K, out, status, stream);
}

}  // namespace pnq
