// pnq_codec_kernels.cu -- dequantize and validate kernels (bit-exact paths).
//
// Dequantize: "PN weight format", section Value (w = d * (n - z), exact in fp32) and
// TandemLLM "Quantisation and profiles", section NVFP4 (e2m1 * e4m3 * global).
// Validate: "PN weight format", section Validation, and NInfer "tensor-formats.md"
// section 3.3 (scale and global validity).
#include "pnq_device.cuh"
#include "pnq_internal.h"

#include <algorithm>
#include <cstdint>

namespace pnq {
namespace {

constexpr int kThreads = 256;

int grid_for(int64_t work_items, int per_thread) {
    const int64_t blocks = (work_items / per_thread + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
    return static_cast<int>(std::max<int64_t>(1, std::min(blocks, cap)));
}

// A warp takes 32 consecutive blocks at a time (1088 bytes in, 32 * BLK floats out). It stages
// the blocks in shared memory, with 16-byte loads when W is 16-byte aligned (16-bit loads
// otherwise: odd blocks start on a 2-byte boundary), then lane l writes float4 j = l, l + 32, ..
// of the chunk's output: elements 4j .. 4j + 3 lie in one block (BLK is a multiple of 4), each a
// code read from its 16-bit half (word e / CPW, half t & 1, shift BITS * (t >> 1), t = e mod CPW)
// times d, exact in fp32. The writes, 9.4 of every 10 bytes moved, are whole 512-byte warp stores.
constexpr int kChunkBlocks = 32;
constexpr int kChunkBytes = kChunkBlocks * kBlockBytes;  // 1088 = 68 * 16

template <int TYPE, bool VEC>
__global__ void __launch_bounds__(kThreads) pn_dequant_kernel(const uint8_t* __restrict__ W, int64_t nblocks,
                                                                float* __restrict__ out) {
    using F = PnFmt<TYPE>;
    __shared__ __align__(16) uint8_t stage[kThreads / 32][kChunkBytes];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* sb = stage[warp];
    const int64_t nchunks = (nblocks + kChunkBlocks - 1) / kChunkBlocks;
    const int64_t wstride = static_cast<int64_t>(gridDim.x) * (kThreads / 32);
    for (int64_t ch = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + warp; ch < nchunks; ch += wstride) {
        const int64_t left = nblocks - ch * kChunkBlocks;
        const int nblk = left < kChunkBlocks ? static_cast<int>(left) : kChunkBlocks;
        const uint8_t* src = W + ch * kChunkBytes;
        if (VEC && nblk == kChunkBlocks) {
            for (int q = lane; q < kChunkBytes / 16; q += 32)
                reinterpret_cast<uint4*>(sb)[q] = __ldg(reinterpret_cast<const uint4*>(src) + q);
        } else {
            for (int q = lane; q < nblk * kBlockBytes / 2; q += 32)
                reinterpret_cast<unsigned short*>(sb)[q] = __ldg(reinterpret_cast<const unsigned short*>(src) + q);
        }
        __syncwarp();
        const int nvec = nblk * F::BLK / 4;
        float4* o = reinterpret_cast<float4*>(out + ch * kChunkBlocks * F::BLK);
        for (int j = lane; j < nvec; j += 32) {
            const int blk = (4 * j) / F::BLK, e0 = 4 * j - blk * F::BLK;
            const uint8_t* bp = sb + blk * kBlockBytes;
            const float d = __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(bp)));
            float v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int e = e0 + q, w = e / F::CPW, t = e - w * F::CPW;
                const uint32_t half = *reinterpret_cast<const unsigned short*>(bp + 2 + 4 * w + 2 * (t & 1));
                const int n = static_cast<int>((half >> (F::BITS * (t >> 1))) & ((1u << F::BITS) - 1u));
                v[q] = __fmul_rn(d, static_cast<float>(n - F::Z));
            }
            if (VEC) {
                o[j] = make_float4(v[0], v[1], v[2], v[3]);
            } else {
                float* os = reinterpret_cast<float*>(o) + 4 * j;
                os[0] = v[0];
                os[1] = v[1];
                os[2] = v[2];
                os[3] = v[3];
            }
        }
        __syncwarp();
    }
}

// One thread per two code bytes (four weights, one float4): code byte c of the flat [N][K/2]
// array belongs to scale c / 8 of the flat [N][K/16] array; a warp writes 512 contiguous bytes.
// A thread takes UNR such pairs a grid stride apart per round, all loads first, so that UNR code
// and scale loads per thread are in flight at once.
constexpr int kNvUnroll = 4;

template <bool DIV, bool VEC>
__global__ void __launch_bounds__(kThreads) nvfp4_dequant_kernel(const uint8_t* __restrict__ codes,
                                                                   const uint8_t* __restrict__ scales, float g,
                                                                   int64_t npairs, float* __restrict__ out) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i0 < npairs;
         i0 += kNvUnroll * stride) {
        uint32_t c[kNvUnroll], sb[kNvUnroll];
#pragma unroll
        for (int u = 0; u < kNvUnroll; ++u) {
            const int64_t i = i0 + u * stride;
            c[u] = 0u;
            sb[u] = 0u;
            if (i < npairs) {
                c[u] = VEC ? __ldg(reinterpret_cast<const unsigned short*>(codes) + i)
                           : (static_cast<uint32_t>(__ldg(codes + 2 * i)) |
                              (static_cast<uint32_t>(__ldg(codes + 2 * i + 1)) << 8));
                sb[u] = __ldg(scales + (i >> 2));
            }
        }
#pragma unroll
        for (int u = 0; u < kNvUnroll; ++u) {
            const int64_t i = i0 + u * stride;
            if (i >= npairs) break;
            const float s = e4m3_to_f32(sb[u]);
            float v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                // e2m1 * e4m3 is exact in fp32; the product with (quotient by) g is the single rounding
                const float p = e2m1_to_f32((c[u] >> (4 * q)) & 15u) * s;
                v[q] = DIV ? __fdiv_rn(p, g) : __fmul_rn(p, g);
            }
            if (VEC) {
                reinterpret_cast<float4*>(out)[i] = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) out[4 * i + q] = v[q];
            }
        }
    }
}

// Staged NVFP4 dequantize for 16-byte aligned codes, scales and output: a warp takes 1024
// consecutive weights at a time (512 code bytes, 64 scale bytes), copies them to shared memory
// with 16-byte loads, then lane l writes float4 j = l, l + 32, .. of the chunk's output: weights
// 4j .. 4j + 3, code bytes 2j and 2j + 1, scale byte j / 4. Every warp load and store covers
// 512 contiguous bytes. Whole chunks only (the caller runs the rest through the kernel above).
constexpr int kNvChunk = 1024;  // weights per warp chunk

template <bool DIV>
__global__ void __launch_bounds__(kThreads) nvfp4_dequant_staged_kernel(const uint8_t* __restrict__ codes,
                                                                          const uint8_t* __restrict__ scales, float g,
                                                                          int64_t nchunks, float* __restrict__ out) {
    __shared__ __align__(16) uint8_t stage[kThreads / 32][kNvChunk / 2 + kNvChunk / 16];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* sb = stage[warp];
    const int64_t wstride = static_cast<int64_t>(gridDim.x) * (kThreads / 32);
    for (int64_t ch = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + warp; ch < nchunks; ch += wstride) {
        reinterpret_cast<uint4*>(sb)[lane] = __ldg(reinterpret_cast<const uint4*>(codes) + ch * 32 + lane);
        if (lane < 4)
            reinterpret_cast<uint4*>(sb + kNvChunk / 2)[lane] = __ldg(reinterpret_cast<const uint4*>(scales) + ch * 4 + lane);
        __syncwarp();
        float4* o = reinterpret_cast<float4*>(out) + ch * (kNvChunk / 4);
#pragma unroll
        for (int k = 0; k < kNvChunk / 4 / 32; ++k) {
            const int j = lane + 32 * k;
            const uint32_t c = *reinterpret_cast<const unsigned short*>(sb + 2 * j);
            const float s = e4m3_to_f32(sb[kNvChunk / 2 + (j >> 2)]);
            float v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                // e2m1 * e4m3 is exact in fp32; the product with (quotient by) g is the single rounding
                const float p = e2m1_to_f32((c >> (4 * q)) & 15u) * s;
                v[q] = DIV ? __fdiv_rn(p, g) : __fmul_rn(p, g);
            }
            o[j] = make_float4(v[0], v[1], v[2], v[3]);
        }
        __syncwarp();
    }
}

// One warp per row. Half h of a row is half h mod 17 of its block (half 0: d, invalid if its
// exponent field is all ones; halves 1..16: word halves, whose bit 15 — word bits 15 and 31 — is
// reserved in pn3t). With 16-byte aligned rows (W aligned, row length a multiple of 16 bytes) a
// lane reads 8 halves per 16-byte load, five loads in flight (a 2,176-byte pn3t row in one round
// trip of the warp), and checks a chunk's halves as four
// 32-bit words: the chunk starting at half 8q holds at most one d, half (17 - 8q mod 17) mod 17
// of the chunk when that is below 8; every other half of a pn3t chunk must have bit 15 clear.
// Otherwise 16-bit loads. Positions mod 17 stay in 32 bits.
constexpr int kValLoads = 5;

template <int TYPE, bool VEC>
__global__ void __launch_bounds__(kThreads) pn_validate_kernel(const uint8_t* __restrict__ W, int64_t n_rows,
                                                                 int row_halves, int32_t* __restrict__ flags) {
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t row = warp0; row < n_rows; row += nwarps) {
        const unsigned short* h = reinterpret_cast<const unsigned short*>(W) + row * row_halves;
        bool bad = false;
        if (VEC) {
            const uint4* v = reinterpret_cast<const uint4*>(h);
            const int nq = row_halves / 8;
            for (int q0 = lane; q0 < nq; q0 += kValLoads * 32) {
                uint4 u[kValLoads];
#pragma unroll
                for (int j = 0; j < kValLoads; ++j) u[j] = (q0 + 32 * j < nq) ? __ldg(v + q0 + 32 * j) : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int j = 0; j < kValLoads; ++j) {
                    const int p0 = (8 * (q0 + 32 * j)) % 17;  // position of the chunk's first half
                    const int hd = p0 == 0 ? 0 : 17 - p0;       // the chunk's d half, if below 8
                    const int wd = hd >> 1;
                    const uint32_t w = wd == 0 ? u[j].x : wd == 1 ? u[j].y : wd == 2 ? u[j].z : u[j].w;
                    // zero chunks past the row are valid halves
                    bad |= hd < 8 && ((w >> (16 * (hd & 1))) & 0x7C00u) == 0x7C00u;
                    if (TYPE == kTypePn3t) {
                        const uint32_t dm = hd < 8 ? ((hd & 1) ? 0x80000000u : 0x00008000u) : 0u;
                        const uint32_t r = (u[j].x & (0x80008000u ^ (wd == 0 ? dm : 0u))) |
                                           (u[j].y & (0x80008000u ^ (wd == 1 ? dm : 0u))) |
                                           (u[j].z & (0x80008000u ^ (wd == 2 ? dm : 0u))) |
                                           (u[j].w & (0x80008000u ^ (wd == 3 ? dm : 0u)));
                        bad |= r != 0u;
                    }
                }
            }
        } else {
            for (int i = lane; i < row_halves; i += 32) {
                const uint32_t x = __ldg(h + i);
                bad |= (i % 17 == 0) ? (x & 0x7C00u) == 0x7C00u : (TYPE == kTypePn3t && (x & 0x8000u) != 0);
            }
        }
        bad = __any_sync(0xffffffffu, bad);
        if (lane == 0) flags[row] = bad ? 1 : 0;
    }
}

// One warp per row of scale bytes: a byte with its sign bit set or the NaN pattern 0x7F / 0xFF
// makes the row invalid, and so does a global field that is not finite and > 0 (g_ok == 0, every
// row). 16 bytes per lane-load when the rows are 16-byte aligned.
template <bool VEC>
__global__ void __launch_bounds__(kThreads) nvfp4_validate_kernel(const uint8_t* __restrict__ scales, int64_t n_rows,
                                                                    int ns, int g_ok, int32_t* __restrict__ flags) {
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    auto bad_byte = [](uint32_t b) { return (b & 0x80u) != 0 || (b & 0x7Fu) == 0x7Fu; };
    for (int64_t row = warp0; row < n_rows; row += nwarps) {
        const uint8_t* r = scales + row * ns;
        bool bad = !g_ok;
        if (g_ok) {
            if (VEC) {
                for (int q = lane; q < ns / 16; q += 32) {
                    const uint4 u = __ldg(reinterpret_cast<const uint4*>(r) + q);
                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int k = 0; k < 16; ++k) bad |= bad_byte((w[k >> 2] >> (8 * (k & 3))) & 0xFFu);
                }
            } else {
                for (int i = lane; i < ns; i += 32) bad |= bad_byte(__ldg(r + i));
            }
        }
        bad = __any_sync(0xffffffffu, bad);
        if (lane == 0) flags[row] = bad ? 1 : 0;
    }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

cudaError_t launch_pn_dequant(int type, const uint8_t* W, int64_t n_rows, int64_t K, float* out,
                              cudaStream_t stream) {
    const int blk = (type == kTypePn3t) ? PnFmt<kTypePn3t>::BLK : PnFmt<kTypePn4t>::BLK;
    const int64_t nblocks = n_rows * (K / blk);
    if (nblocks == 0) return cudaSuccess;
    const int grid = grid_for((nblocks + kChunkBlocks - 1) / kChunkBlocks * 32, 1);
    const bool vec = aligned16(W) && aligned16(out);
    if (type == kTypePn3t) {
        if (vec) pn_dequant_kernel<kTypePn3t, true><<<grid, kThreads, 0, stream>>>(W, nblocks, out);
        else pn_dequant_kernel<kTypePn3t, false><<<grid, kThreads, 0, stream>>>(W, nblocks, out);
    } else {
        if (vec) pn_dequant_kernel<kTypePn4t, true><<<grid, kThreads, 0, stream>>>(W, nblocks, out);
        else pn_dequant_kernel<kTypePn4t, false><<<grid, kThreads, 0, stream>>>(W, nblocks, out);
    }
    return cudaGetLastError();
}

// NVFP4 dequantize of npairs code-byte pairs from w's pointers, by the pair-per-thread kernel.
cudaError_t launch_nvfp4_dequant_pairs(const Nvfp4View& w, int64_t npairs, float* out, cudaStream_t stream);

cudaError_t launch_nvfp4_dequant(const Nvfp4View& w, int64_t n_rows, int64_t K, float* out,
                                 cudaStream_t stream) {
    const int64_t npairs = n_rows * (K / 4);
    if (npairs == 0) return cudaSuccess;
    // whole 1024-weight chunks through the staged kernel when everything is 16-byte aligned
    if (aligned16(w.codes) && aligned16(w.scales) && aligned16(out)) {
        const int64_t nchunks = npairs * 4 / kNvChunk;
        if (nchunks > 0) {
            const int g2 = grid_for(nchunks * 32, 1);
            if (w.div)
                nvfp4_dequant_staged_kernel<true><<<g2, kThreads, 0, stream>>>(w.codes, w.scales, w.g, nchunks, out);
            else
                nvfp4_dequant_staged_kernel<false><<<g2, kThreads, 0, stream>>>(w.codes, w.scales, w.g, nchunks, out);
            const cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return e;
        }
        const int64_t done = nchunks * kNvChunk;  // weights written
        const int64_t rest = npairs - done / 4;
        if (rest == 0) return cudaSuccess;
        Nvfp4View tail = w;
        tail.codes = w.codes + done / 2;
        tail.scales = w.scales + done / 16;
        return launch_nvfp4_dequant_pairs(tail, rest, out + done, stream);
    }
    return launch_nvfp4_dequant_pairs(w, npairs, out, stream);
}

cudaError_t launch_nvfp4_dequant_pairs(const Nvfp4View& w, int64_t npairs, float* out, cudaStream_t stream) {
    const int grid = grid_for(npairs, kNvUnroll);
    const bool vec = (reinterpret_cast<uintptr_t>(w.codes) & 1u) == 0 && aligned16(out);
    if (w.div) {
        if (vec) nvfp4_dequant_kernel<true, true><<<grid, kThreads, 0, stream>>>(w.codes, w.scales, w.g, npairs, out);
        else nvfp4_dequant_kernel<true, false><<<grid, kThreads, 0, stream>>>(w.codes, w.scales, w.g, npairs, out);
    } else {
        if (vec) nvfp4_dequant_kernel<false, true><<<grid, kThreads, 0, stream>>>(w.codes, w.scales, w.g, npairs, out);
        else nvfp4_dequant_kernel<false, false><<<grid, kThreads, 0, stream>>>(w.codes, w.scales, w.g, npairs, out);
    }
    return cudaGetLastError();
}

cudaError_t launch_pn_validate(int type, const uint8_t* W, int64_t n_rows, int64_t K, int32_t* flags,
                               cudaStream_t stream) {
    if (n_rows == 0) return cudaSuccess;
    const int blk = (type == kTypePn3t) ? PnFmt<kTypePn3t>::BLK : PnFmt<kTypePn4t>::BLK;
    const int64_t nb = K / blk;
    if (nb * 17 > INT32_MAX) return cudaErrorInvalidValue;  // rows of over 2^31 halves
    const int row_halves = static_cast<int>(nb * 17);
    const bool vec = aligned16(W) && (nb * kBlockBytes) % 16 == 0;
    const int grid = grid_for(n_rows * 32, 1);
    if (type == kTypePn3t) {
        if (vec) pn_validate_kernel<kTypePn3t, true><<<grid, kThreads, 0, stream>>>(W, n_rows, row_halves, flags);
        else pn_validate_kernel<kTypePn3t, false><<<grid, kThreads, 0, stream>>>(W, n_rows, row_halves, flags);
    } else {
        if (vec) pn_validate_kernel<kTypePn4t, true><<<grid, kThreads, 0, stream>>>(W, n_rows, row_halves, flags);
        else pn_validate_kernel<kTypePn4t, false><<<grid, kThreads, 0, stream>>>(W, n_rows, row_halves, flags);
    }
    return cudaGetLastError();
}

cudaError_t launch_nvfp4_validate(const Nvfp4View& w, int64_t n_rows, int64_t K, int32_t* flags,
                                  cudaStream_t stream) {
    if (n_rows == 0) return cudaSuccess;
    const int g_ok = (w.g > 0.0f && w.g <= 3.4028234663852886e38f) ? 1 : 0;  // finite and > 0
    if (K / 16 > INT32_MAX) return cudaErrorInvalidValue;  // rows of over 2^31 scales
    const int ns = static_cast<int>(K / 16);
    const bool vec = aligned16(w.scales) && ns % 16 == 0;
    const int grid = grid_for(n_rows * 32, 1);
    if (vec) nvfp4_validate_kernel<true><<<grid, kThreads, 0, stream>>>(w.scales, n_rows, ns, g_ok, flags);
    else nvfp4_validate_kernel<false><<<grid, kThreads, 0, stream>>>(w.scales, n_rows, ns, g_ok, flags);
    return cudaGetLastError();
}

}  // namespace pnq
