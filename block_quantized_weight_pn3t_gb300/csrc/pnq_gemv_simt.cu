// pnq_gemv_simt.cu -- generic GEMV path (CUDA-core fp32 FMA, any alignment).
//
// Y[m][n] = sum_k w[n][k] x[m][k] with w decoded as on the "PN weight format" page
// (section Value) or as TandemLLM's NVFP4 (e2m1 * e4m3 * global). It takes every layout the
// C ABI accepts -- PN rows at any 2-byte alignment and any K that is a multiple of the block
// size, NVFP4 at any K that is a multiple of 16 -- and is the reference point the tensor-core
// path is measured against. One warp per output row; lanes stride over blocks (PN) or
// 16-weight groups (NVFP4); each block's sum over its weights is formed first and scaled
// once by the block's scale.
#include "pnq_device.cuh"
#include "pnq_internal.h"

#include <algorithm>

namespace pnq {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxM = 16;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int TYPE>
__global__ void __launch_bounds__(kThreads) pn_gemv_simt_kernel(const uint8_t* __restrict__ W, int64_t N,
                                                                  int64_t K, const float* __restrict__ X, int M,
                                                                  float* __restrict__ Y) {
    using F = PnFmt<TYPE>;
    const int lane = threadIdx.x & 31;
    const int64_t nb = K / F::BLK;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t row = warp0; row < N; row += nwarps) {
        float acc[kMaxM];
#pragma unroll
        for (int m = 0; m < kMaxM; ++m) acc[m] = 0.0f;
        const uint8_t* rowp = W + row * nb * kBlockBytes;
        for (int64_t b = lane; b < nb; b += 32) {
            const uint8_t* blk = rowp + b * kBlockBytes;
            const float d = __half2float(__ushort_as_half(__ldg(reinterpret_cast<const unsigned short*>(blk))));
            float s[kMaxM];
#pragma unroll
            for (int m = 0; m < kMaxM; ++m) s[m] = 0.0f;
            const float* xb = X + b * F::BLK;
#pragma unroll 1
            for (int h = 0; h < 16; ++h) {  // 16-bit half h: word h/2, even t (h even) or odd t
                const uint32_t half = __ldg(reinterpret_cast<const unsigned short*>(blk + 2 + 2 * h));
                const int e0 = (h >> 1) * F::CPW + (h & 1);
#pragma unroll
                for (int j = 0; j < F::PAIRS; ++j) {
                    const float q = static_cast<float>(
                        static_cast<int>((half >> (F::BITS * j)) & ((1u << F::BITS) - 1u)) - F::Z);
                    const int e = e0 + 2 * j;
#pragma unroll
                    for (int m = 0; m < kMaxM; ++m)
                        if (m < M) s[m] = fmaf(q, __ldg(xb + m * K + e), s[m]);
                }
            }
#pragma unroll
            for (int m = 0; m < kMaxM; ++m) acc[m] = fmaf(d, s[m], acc[m]);
        }
#pragma unroll
        for (int m = 0; m < kMaxM; ++m) {
            if (m < M) {
                const float v = warp_sum(acc[m]);
                if (lane == 0) Y[m * N + row] = v;
            }
        }
    }
}

// g multiplies each output, or divides it (div: the divisor reading of the global field).
__global__ void __launch_bounds__(kThreads) nvfp4_gemv_simt_kernel(const uint8_t* __restrict__ codes,
                                                                     const uint8_t* __restrict__ scales, float g,
                                                                     bool div, int64_t N, int64_t K,
                                                                     const uint16_t* __restrict__ X, int M,
                                                                     float* __restrict__ Y) {
    const int lane = threadIdx.x & 31;
    const int64_t ng = K / 16;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t row = warp0; row < N; row += nwarps) {
        float acc[kMaxM];
#pragma unroll
        for (int m = 0; m < kMaxM; ++m) acc[m] = 0.0f;
        for (int64_t grp = lane; grp < ng; grp += 32) {
            const float sc = e4m3_to_f32(__ldg(scales + row * ng + grp));
            float s[kMaxM];
#pragma unroll
            for (int m = 0; m < kMaxM; ++m) s[m] = 0.0f;
            const uint8_t* cp = codes + row * (K / 2) + grp * 8;
            const uint16_t* xg = X + grp * 16;
#pragma unroll 1
            for (int q = 0; q < 8; ++q) {
                const uint32_t c = __ldg(cp + q);
                const float v0 = e2m1_to_f32(c & 15u), v1 = e2m1_to_f32(c >> 4);
#pragma unroll
                for (int m = 0; m < kMaxM; ++m) {
                    if (m < M) {
                        const float x0 = __uint_as_float(static_cast<uint32_t>(__ldg(xg + m * K + 2 * q)) << 16);
                        const float x1 = __uint_as_float(static_cast<uint32_t>(__ldg(xg + m * K + 2 * q + 1)) << 16);
                        s[m] = fmaf(v1, x1, fmaf(v0, x0, s[m]));
                    }
                }
            }
#pragma unroll
            for (int m = 0; m < kMaxM; ++m) acc[m] = fmaf(sc, s[m], acc[m]);
        }
#pragma unroll
        for (int m = 0; m < kMaxM; ++m) {
            if (m < M) {
                const float v = warp_sum(acc[m]);
                if (lane == 0) Y[m * N + row] = div ? v / g : v * g;
            }
        }
    }
}

int rows_grid(int64_t N) {
    const int64_t blocks = (N * 32 + kThreads - 1) / kThreads;
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(blocks, int64_t(device_sm_count()) * 16)));
}

}  // namespace

cudaError_t launch_pn_gemv_simt(int type, const uint8_t* W, int64_t N, int64_t K, const float* X, int M,
                                float* Y, cudaStream_t stream) {
    if (N == 0) return cudaSuccess;
    if (type == kTypePn3t)
        pn_gemv_simt_kernel<kTypePn3t><<<rows_grid(N), kThreads, 0, stream>>>(W, N, K, X, M, Y);
    else
        pn_gemv_simt_kernel<kTypePn4t><<<rows_grid(N), kThreads, 0, stream>>>(W, N, K, X, M, Y);
    return cudaGetLastError();
}

cudaError_t launch_nvfp4_gemv_simt(const Nvfp4View& w, int64_t N, int64_t K, const uint16_t* X, int M,
                                   float* Y, cudaStream_t stream) {
    if (N == 0) return cudaSuccess;
    nvfp4_gemv_simt_kernel<<<rows_grid(N), kThreads, 0, stream>>>(w.codes, w.scales, w.g, w.div, N, K, X, M, Y);
    return cudaGetLastError();
}

}  // namespace pnq
