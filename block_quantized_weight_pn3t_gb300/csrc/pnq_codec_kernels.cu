// pnq_codec_kernels.cu -- dequantize and validate kernels (bit-exact paths).
//
// Dequantize: "PN weight format", section Value (w = d * (n - z), exact in fp32) and
// TandemLLM "Quantisation and profiles", section NVFP4 (e2m1 * e4m3 * global).
// Validate: "PN weight format", section Validation, and NInfer "tensor-formats.md"
// section 3.3 (scale and global validity).
#include "pnq_device.cuh"
#include "pnq_internal.h"

#include <algorithm>

namespace pnq {
namespace {

constexpr int kThreads = 256;

int grid_for(int64_t work_items, int per_thread) {
    const int64_t blocks = (work_items / per_thread + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
    return static_cast<int>(std::max<int64_t>(1, std::min(blocks, cap)));
}

// One thread per (block, 16-bit half): the half holds the codes of CPW/2 elements, all
// even t (low half of a word) or all odd t (high half); only 16-bit loads are used, so
// the 2-byte alignment of odd blocks is never an issue. Output row-major order equals
// block order, so block gb writes out[gb * BLK + e].
template <int TYPE>
__global__ void __launch_bounds__(kThreads) pn_dequant_kernel(const uint8_t* __restrict__ W, int64_t nblocks,
                                                                float* __restrict__ out) {
    using F = PnFmt<TYPE>;
    const int64_t total = nblocks * 16;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t gb = i >> 4;
        const int h = static_cast<int>(i & 15);
        const uint8_t* blk = W + gb * kBlockBytes;
        const float d = __half2float(__ushort_as_half(__ldg(reinterpret_cast<const unsigned short*>(blk))));
        const uint32_t half = __ldg(reinterpret_cast<const unsigned short*>(blk + 2 + 2 * h));
        float* o = out + gb * F::BLK + (h >> 1) * F::CPW + (h & 1);
#pragma unroll
        for (int j = 0; j < F::PAIRS; ++j) {
            const int n = static_cast<int>((half >> (F::BITS * j)) & ((1u << F::BITS) - 1u));
            o[2 * j] = d * static_cast<float>(n - F::Z);
        }
    }
}

// One thread per code byte (two weights); code byte c of the flat [N][K/2] array belongs
// to scale c / 8 of the flat [N][K/16] array.
template <bool DIV>
__global__ void __launch_bounds__(kThreads) nvfp4_dequant_kernel(const uint8_t* __restrict__ codes,
                                                                   const uint8_t* __restrict__ scales, float g,
                                                                   int64_t nbytes, float* __restrict__ out) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nbytes; i += stride) {
        const uint32_t c = __ldg(codes + i);
        const float s = e4m3_to_f32(__ldg(scales + (i >> 3)));
        // e2m1 * e4m3 is exact in fp32; the product with (quotient by) g is the single rounding.
        const float lo = e2m1_to_f32(c & 15u) * s;
        const float hi = e2m1_to_f32(c >> 4) * s;
        out[2 * i] = DIV ? __fdiv_rn(lo, g) : __fmul_rn(lo, g);
        out[2 * i + 1] = DIV ? __fdiv_rn(hi, g) : __fmul_rn(hi, g);
    }
}

// One warp per row over the row's 16-bit halves: half 0 of each 17-half block is d
// (invalid if its exponent field is all ones), the other 16 are word halves whose bit 15
// (word bits 15 and 31) is reserved in pn3t.
template <int TYPE>
__global__ void __launch_bounds__(kThreads) pn_validate_kernel(const uint8_t* __restrict__ W, int64_t n_rows,
                                                                 int64_t nb, int32_t* __restrict__ flags) {
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t nh = nb * 17;
    for (int64_t row = warp0; row < n_rows; row += nwarps) {
        const unsigned short* h = reinterpret_cast<const unsigned short*>(W + row * nb * kBlockBytes);
        bool bad = false;
        int pos = lane % 17;
        for (int64_t i = lane; i < nh; i += 32) {
            const uint32_t v = __ldg(h + i);
            if (pos == 0)
                bad |= (v & 0x7C00u) == 0x7C00u;
            else if (TYPE == kTypePn3t)
                bad |= (v & 0x8000u) != 0;
            pos += 15;  // (i + 32) mod 17
            if (pos >= 17) pos -= 17;
        }
        bad = __any_sync(0xffffffffu, bad);
        if (lane == 0) flags[row] = bad ? 1 : 0;
    }
}

__global__ void __launch_bounds__(kThreads) nvfp4_validate_kernel(const uint8_t* __restrict__ scales,
                                                                    int64_t n_rows, int64_t ns, int g_ok,
                                                                    int32_t* __restrict__ flags) {
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t row = warp0; row < n_rows; row += nwarps) {
        bool bad = !g_ok;
        for (int64_t i = lane; i < ns; i += 32) {
            const uint32_t s = __ldg(scales + row * ns + i);
            bad |= (s & 0x80u) != 0 || (s & 0x7Fu) == 0x7Fu;
        }
        bad = __any_sync(0xffffffffu, bad);
        if (lane == 0) flags[row] = bad ? 1 : 0;
    }
}

}  // namespace

cudaError_t launch_pn_dequant(int type, const uint8_t* W, int64_t n_rows, int64_t K, float* out,
                              cudaStream_t stream) {
    const int blk = (type == kTypePn3t) ? PnFmt<kTypePn3t>::BLK : PnFmt<kTypePn4t>::BLK;
    const int64_t nblocks = n_rows * (K / blk);
    if (nblocks == 0) return cudaSuccess;
    const int grid = grid_for(nblocks * 16, 1);
    if (type == kTypePn3t)
        pn_dequant_kernel<kTypePn3t><<<grid, kThreads, 0, stream>>>(W, nblocks, out);
    else
        pn_dequant_kernel<kTypePn4t><<<grid, kThreads, 0, stream>>>(W, nblocks, out);
    return cudaGetLastError();
}

cudaError_t launch_nvfp4_dequant(const Nvfp4View& w, int64_t n_rows, int64_t K, float* out,
                                 cudaStream_t stream) {
    const int64_t nbytes = n_rows * (K / 2);
    if (nbytes == 0) return cudaSuccess;
    if (w.div)
        nvfp4_dequant_kernel<true><<<grid_for(nbytes, 1), kThreads, 0, stream>>>(w.codes, w.scales, w.g, nbytes, out);
    else
        nvfp4_dequant_kernel<false><<<grid_for(nbytes, 1), kThreads, 0, stream>>>(w.codes, w.scales, w.g, nbytes, out);
    return cudaGetLastError();
}

cudaError_t launch_pn_validate(int type, const uint8_t* W, int64_t n_rows, int64_t K, int32_t* flags,
                               cudaStream_t stream) {
    if (n_rows == 0) return cudaSuccess;
    const int blk = (type == kTypePn3t) ? PnFmt<kTypePn3t>::BLK : PnFmt<kTypePn4t>::BLK;
    const int grid = grid_for(n_rows * 32, 1);
    if (type == kTypePn3t)
        pn_validate_kernel<kTypePn3t><<<grid, kThreads, 0, stream>>>(W, n_rows, K / blk, flags);
    else
        pn_validate_kernel<kTypePn4t><<<grid, kThreads, 0, stream>>>(W, n_rows, K / blk, flags);
    return cudaGetLastError();
}

cudaError_t launch_nvfp4_validate(const Nvfp4View& w, int64_t n_rows, int64_t K, int32_t* flags,
                                  cudaStream_t stream) {
    if (n_rows == 0) return cudaSuccess;
    const int g_ok = (w.g > 0.0f && w.g <= 3.4028234663852886e38f) ? 1 : 0;  // finite and > 0
    nvfp4_validate_kernel<<<grid_for(n_rows * 32, 1), kThreads, 0, stream>>>(w.scales, n_rows, K / 16, g_ok,
                                                                              flags);
    return cudaGetLastError();
}

}  // namespace pnq
