// pnq_prefill.cu -- PN (pn3t / pn4t) products for more than 16 activation rows (prefill), on the
// fifth-generation tensor cores (tcgen05), sm_103a.
//
// Y[m][n] = sum_k w[n][k] x[m][k] for any M, following the prefill route of the pages (the
// feedman.me post on the BF16_P12 format, section "How the engine uses it": with more than 16
// tokens a cache-sized piece of the weights is unpacked, then multiplied densely).
//
// Exactness. A decoded PN weight d * (n - z) has at most 15 significant bits (11 of the fp16 d
// times a code difference of at most 4 bits), so it is the exact sum of two tf32 numbers:
// w_hi = w with its low 13 fraction bits cleared, w_lo = w - w_hi (at most 4 bits). x is split
// the same way (x_lo keeps the next 11 bits; 2^-22 of |x| is dropped). The product is taken as
// w_hi x_hi + w_hi x_lo + w_lo x_hi, three tf32 MMAs into one fp32 accumulator, dropping only
// w_lo x_lo (2^-22 of |w x|): the GEMV accuracy bound holds.
//
// Pipeline per call: x is split once into two fp32 planes; then, slice by slice of `rows` weight
// rows (as many as the caller's scratch holds, a multiple of 128), the slice is decoded into two
// fp32 planes and multiplied by the GEMM kernel below. Scratch layout: x_hi, x_lo [M][K], then
// w_hi, w_lo [rows][K], all fp32.
//
// GEMM kernel: one CTA per (128 weight rows, BN activation rows) tile. Warp 0 (one thread) loads
// the four operand tiles of each 32-wide K step with 2-D tensor-map copies (128-byte swizzle)
// into a ring of S stages; warp 1 allocates the tensor-memory accumulator (128 lanes x BN fp32
// columns) and one of its threads issues per K step the 3 x 4 tcgen05.mma (kind::tf32, K = 8
// each) and commits them to the stage's "empty" barrier; warps 2..5 read the accumulator back
// (tcgen05.ld, one weight row per thread) and store Y transposed (consecutive threads write
// consecutive n). Every wait is bounded; a wait that gives up records its site in the device
// error word, and the MMA thread always commits the final barrier, so the epilogue and the
// tensor-memory release happen whatever the outcome.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>

#include "pnq_device.cuh"
#include "pnq_internal.h"

namespace pnq {
namespace {

constexpr int kTM = 128;                  // weight rows per tile (MMA M)
constexpr int kTK = 32;                   // K per stage: 32 fp32 = one 128-byte swizzle row
constexpr int kATile = kTM * kTK * 4;     // 16 KB
constexpr int kGemmThreads = 192;         // producer, MMA, four epilogue warps
constexpr size_t kGemmSmemLimit = 227u * 1024u;

// Clears the low 13 fraction bits: the tf32 part of an fp32 value (exact split w = hi + (w - hi)).
__device__ __forceinline__ float tf32_hi(float v) { return __uint_as_float(__float_as_uint(v) & 0xFFFFE000u); }

// x [M][K] -> x_hi, x_lo planes (4 elements per thread).
__global__ void __launch_bounds__(256) split_x_kernel(const float4* __restrict__ x, int64_t n4, float4* __restrict__ hi,
                                                      float4* __restrict__ lo) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
        const float4 v = __ldg(x + i);
        const float4 h = make_float4(tf32_hi(v.x), tf32_hi(v.y), tf32_hi(v.z), tf32_hi(v.w));
        hi[i] = h;
        lo[i] = make_float4(v.x - h.x, v.y - h.y, v.z - h.z, v.w - h.w);
    }
}

// A slice of consecutive PN blocks (whole rows) -> w_hi, w_lo planes in the same element order.
// A warp takes 32 blocks at a time (1088 bytes): it stages them in shared memory (16-byte loads
// when the chunk is 16-byte aligned, 16-bit loads otherwise), then lane l decodes elements
// 4j .. 4j + 3 (one block: BLK is a multiple of 4) for j = l, l + 32, .. and writes one float4 to
// each plane, so every warp store covers 512 contiguous bytes.
constexpr int kSliceChunk = 32;
constexpr int kSliceChunkBytes = kSliceChunk * kBlockBytes;  // 1088 = 68 * 16

template <int TYPE, bool VEC>
__global__ void __launch_bounds__(256) decode_slice_kernel(const uint8_t* __restrict__ W, int64_t nblocks,
                                                           float* __restrict__ hi, float* __restrict__ lo) {
    using F = PnFmt<TYPE>;
    __shared__ __align__(16) uint8_t stage[8][kSliceChunkBytes];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* sb = stage[warp];
    const int64_t nchunks = (nblocks + kSliceChunk - 1) / kSliceChunk;
    const int64_t wstride = static_cast<int64_t>(gridDim.x) * 8;
    for (int64_t ch = static_cast<int64_t>(blockIdx.x) * 8 + warp; ch < nchunks; ch += wstride) {
        const int64_t left = nblocks - ch * kSliceChunk;
        const int nblk = left < kSliceChunk ? static_cast<int>(left) : kSliceChunk;
        const uint8_t* src = W + ch * kSliceChunkBytes;
        if (VEC && nblk == kSliceChunk) {
            for (int q = lane; q < kSliceChunkBytes / 16; q += 32)
                reinterpret_cast<uint4*>(sb)[q] = __ldg(reinterpret_cast<const uint4*>(src) + q);
        } else {
            for (int q = lane; q < nblk * kBlockBytes / 2; q += 32)
                reinterpret_cast<unsigned short*>(sb)[q] = __ldg(reinterpret_cast<const unsigned short*>(src) + q);
        }
        __syncwarp();
        const int nvec = nblk * F::BLK / 4;
        float4* oh = reinterpret_cast<float4*>(hi + ch * kSliceChunk * F::BLK);
        float4* ol = reinterpret_cast<float4*>(lo + ch * kSliceChunk * F::BLK);
        for (int j = lane; j < nvec; j += 32) {
            const int blk = (4 * j) / F::BLK, e0 = 4 * j - blk * F::BLK;
            const uint8_t* bp = sb + blk * kBlockBytes;
            const float d = __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(bp)));
            float v[4], h[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int e = e0 + q, w = e / F::CPW, t = e - w * F::CPW;
                const uint32_t half = *reinterpret_cast<const unsigned short*>(bp + 2 + 4 * w + 2 * (t & 1));
                const int n = static_cast<int>((half >> (F::BITS * (t >> 1))) & ((1u << F::BITS) - 1u));
                v[q] = d * static_cast<float>(n - F::Z);  // exact in fp32
                h[q] = tf32_hi(v[q]);
            }
            oh[j] = make_float4(h[0], h[1], h[2], h[3]);
            ol[j] = make_float4(v[0] - h[0], v[1] - h[1], v[2] - h[2], v[3] - h[3]);
        }
        __syncwarp();
    }
}

template <int TYPE>
void launch_decode_slice(const uint8_t* W, int64_t nblocks, float* hi, float* lo, int sms, cudaStream_t stream) {
    const int64_t chunks = (nblocks + kSliceChunk - 1) / kSliceChunk;
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((chunks + 7) / 8, int64_t(sms) * 8)));
    if (reinterpret_cast<uintptr_t>(W) % 16 == 0)
        decode_slice_kernel<TYPE, true><<<grid, 256, 0, stream>>>(W, nblocks, hi, lo);
    else
        decode_slice_kernel<TYPE, false><<<grid, 256, 0, stream>>>(W, nblocks, hi, lo);
}

// Shared-memory matrix descriptor, K-major with the 128-byte swizzle (rows of 128 bytes, 8-row
// groups 1024 bytes apart); the tile starts on a 1024-byte boundary, and the K steps inside a
// swizzle row advance the start address by their byte offset.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
    return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (1ull << 16) | (static_cast<uint64_t>(1024 >> 4) << 32) |
           (1ull << 46) | (2ull << 61);
}

// D (tensor memory, f32) [+]= A (shared, tf32, K-major) x B (shared, tf32, K-major); one thread.
__device__ __forceinline__ void mma_tf32_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

struct GemmArgs {
    float* Y;
    int* err;
    int M, rows, K, S;  // activation rows, weight rows of the slice, K, stages
    int ks;             // K split over a cluster of ks CTAs along z (1: none)
    int64_t ldy, n0;    // Y row stride (N) and the slice's first weight row
};

template <int BN>
__global__ void __launch_bounds__(kGemmThreads, 1) tf32_gemm_kernel(const __grid_constant__ CUtensorMap mwh,
                                                                     const __grid_constant__ CUtensorMap mwl,
                                                                     const __grid_constant__ CUtensorMap mxh,
                                                                     const __grid_constant__ CUtensorMap mxl,
                                                                     const GemmArgs a) {
    constexpr int kBTile = BN * kTK * 4;
    constexpr int kStage = 2 * kATile + 2 * kBTile;
    constexpr uint32_t kCols = BN < 32 ? 32 : BN;  // tensor-memory columns (a power of two)
    // instruction descriptor: D f32, A and B tf32, both K-major, N = BN, M = 128
    constexpr uint32_t kIdesc = (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
                                (static_cast<uint32_t>(kTM >> 4) << 24);
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    __shared__ __align__(8) uint64_t bars[2 * 8 + 1];
    __shared__ uint32_t tmem_slot;
    const int S = a.S;
    const uint32_t b0 = smem_addr(bars);
    auto full = [&](int s) { return b0 + 8u * s; };
    auto empty = [&](int s) { return b0 + 8u * (8 + s); };
    const uint32_t done = b0 + 8u * 16;
    auto stage = [&](int s) { return smem_addr(base) + static_cast<uint32_t>(s * kStage); };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = blockIdx.x * kTM, col0 = blockIdx.y * BN;
    // this CTA's K tiles [kt0, kt0 + nk): share blockIdx.z of a.ks (every share holds at least one)
    const int nk_all = (a.K + kTK - 1) / kTK, kz = static_cast<int>(blockIdx.z);
    const int kt0 = kz * nk_all / a.ks, nk = (kz + 1) * nk_all / a.ks - kt0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        mbar_init(done, 1);
        mbar_fence_init();
    }
    if (warp == 1) tmem_alloc(smem_addr(&tmem_slot), kCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_w = l2_policy_evict_first(), pol_x = l2_policy_evict_last();
            bool ok = true;
            int kt = 0;
            for (; kt < nk; ++kt) {
                const int s = kt % S;
                if (kt >= S && !mbar_wait_bounded(empty(s), ((kt / S) - 1) & 1)) {
                    ok = false;
                    break;
                }
                const uint32_t st = stage(s);
                const int kx = (kt0 + kt) * kTK;
                mbar_arrive_expect_tx(full(s), static_cast<uint32_t>(kStage));
                tma_load_2d(st, &mwh, kx, row0, full(s), pol_w);
                tma_load_2d(st + kATile, &mwl, kx, row0, full(s), pol_w);
                tma_load_2d(st + 2 * kATile, &mxh, kx, col0, full(s), pol_x);
                tma_load_2d(st + 2 * kATile + kBTile, &mxl, kx, col0, full(s), pol_x);
            }
            if (!ok) record_error(a.err, kErrEmptyWait);
            bool drained = true;  // every copy issued has landed before the CTA may exit
            for (int g = max(0, kt - S); drained && g < kt; ++g) drained = mbar_wait_bounded(full(g % S), (g / S) & 1);
            if (!drained) record_error(a.err, kErrDrainWait);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            bool ok = true;
            for (int kt = 0; kt < nk && ok; ++kt) {
                const int s = kt % S;
                if (!mbar_wait_bounded(full(s), (kt / S) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t st = stage(s);
#pragma unroll
                for (int kk = 0; kk < kTK / 8; ++kk) {  // K = 8 tf32 = 32 bytes per MMA
                    const uint64_t ah = desc_sw128(st + 32 * kk), al = desc_sw128(st + kATile + 32 * kk);
                    const uint64_t bh = desc_sw128(st + 2 * kATile + 32 * kk);
                    const uint64_t bl = desc_sw128(st + 2 * kATile + kBTile + 32 * kk);
                    mma_tf32_ss(tmem, ah, bh, kIdesc, (kt > 0 || kk > 0) ? 1u : 0u);
                    mma_tf32_ss(tmem, ah, bl, kIdesc, 1u);
                    mma_tf32_ss(tmem, al, bh, kIdesc, 1u);
                }
                tc_commit(empty(s));  // the stage is free once these MMAs have read it
            }
            if (!ok) record_error(a.err, kErrFullWait);
            tc_commit(done);  // always: the epilogue and the release wait for it
        }
    } else {
        // epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. + 31 = weight rows of the tile
        const int q = warp & 3;
        const int r = row0 + 32 * q + lane;  // weight row in the slice
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(done, 0));  // warp-uniform: tcgen05.ld is .aligned
        tc_fence_after();
        if (!ok) {
            if (lane == 0) record_error(a.err, kErrFullWait);
        } else if (a.ks == 1) {
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 16) {
                uint32_t v[16];
                tmem_ld<16>(tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(c0), v);
                tmem_wait_ld();
                if (r < a.rows) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int m = col0 + c0 + j;
                        if (m < a.M) a.Y[static_cast<int64_t>(m) * a.ldy + a.n0 + r] = __uint_as_float(v[j]);
                    }
                }
            }
        } else {
            // the partial tile to shared memory (the stages are free: every MMA has completed),
            // rows kRedPitch floats apart
            float* red = reinterpret_cast<float*>(base);
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 16) {
                uint32_t v[16];
                tmem_ld<16>(tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(c0), v);
                tmem_wait_ld();
                float4* dst = reinterpret_cast<float4*>(red + (32 * q + lane) * (BN + 4) + c0);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    dst[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                         __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    if (a.ks > 1) {
        // CTA kz of the cluster sums its share of the tile's rows over the ks partial tiles, in
        // CTA order (distributed shared memory), and writes Y
        cluster_sync();
        const int share = kTM / a.ks + (kTM % a.ks ? 1 : 0);
        const int rl0 = kz * share, rl1 = min(kTM, rl0 + share);
        const uint32_t rbase = smem_addr(base);
        for (int e = static_cast<int>(threadIdx.x); e < (rl1 - rl0) * BN; e += kGemmThreads) {
            const int rl = rl0 + e % (rl1 - rl0), c = e / (rl1 - rl0);
            const uint32_t off = 4u * static_cast<uint32_t>(rl * (BN + 4) + c);
            float v = 0.0f;
            for (int z = 0; z < a.ks; ++z) v += ld_dsmem_f32(rbase + off, static_cast<uint32_t>(z));
            const int r = row0 + rl, m = col0 + c;
            if (r < a.rows && m < a.M) a.Y[static_cast<int64_t>(m) * a.ldy + a.n0 + r] = v;
        }
        cluster_sync();  // no CTA leaves while another still reads its tile
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kCols);
    }
}

template <int BN>
cudaError_t launch_gemm_bn(const CUtensorMap (&maps)[4], const GemmArgs& a0, cudaStream_t stream) {
    constexpr int kStage = 2 * kATile + 2 * BN * kTK * 4;
    GemmArgs a = a0;
    a.S = static_cast<int>(std::min<size_t>(8, (kGemmSmemLimit - 1024 - 1024) / kStage));
    if (a.S < 2) return cudaErrorNotSupported;
    // the stages also hold a K-split cluster's partial tile (128 rows of BN + 4 floats)
    if (a.ks > 1 && static_cast<size_t>(a.S) * kStage < static_cast<size_t>(kTM) * (BN + 4) * 4) return cudaErrorNotSupported;
    const int smem = a.S * kStage + 1024;
    auto kern = tf32_gemm_kernel<BN>;
    static std::atomic<bool> opted[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!opted[dev].load(std::memory_order_relaxed)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        opted[dev].store(true, std::memory_order_relaxed);
    }
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3((a.rows + kTM - 1) / kTM, (a.M + BN - 1) / BN, a.ks);
    lc.blockDim = dim3(kGemmThreads, 1, 1);
    lc.dynamicSmemBytes = smem;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = static_cast<unsigned>(a.ks);
    lc.attrs = attr;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, kern, maps[0], maps[1], maps[2], maps[3], a);
}

}  // namespace

int64_t prefill_slice_rows(int64_t N, int64_t K, int64_t M, size_t scratch_bytes) {
    const int64_t xb = 8 * M * K;
    if (static_cast<int64_t>(scratch_bytes) < xb) return 0;
    int64_t rows = (static_cast<int64_t>(scratch_bytes) - xb) / (8 * K);
    rows = rows / kTM * kTM;
    const int64_t need = (N + kTM - 1) / kTM * kTM;
    return std::min(rows, need);
}

cudaError_t launch_pn_prefill(int type, const uint8_t* W, int64_t N, int64_t K, const float* X, int64_t M, float* Y,
                              int* err, void* scratch, size_t scratch_bytes, cudaStream_t stream) {
    const int blk = (type == kTypePn3t) ? PnFmt<kTypePn3t>::BLK : PnFmt<kTypePn4t>::BLK;
    const int64_t nb = K / blk;
    const int64_t rows = prefill_slice_rows(N, K, M, scratch_bytes);
    if (rows < kTM) return cudaErrorMemoryAllocation;  // the caller's scratch is too small
    float* xh = static_cast<float*>(scratch);
    float* xl = xh + M * K;
    float* wh = xl + M * K;
    float* wl = wh + rows * K;
    const int sms = device_sm_count();
    {
        const int64_t n4 = M * K / 4;
        const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((n4 + 255) / 256, int64_t(sms) * 16)));
        split_x_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<const float4*>(X), n4, reinterpret_cast<float4*>(xh),
                                                 reinterpret_cast<float4*>(xl));
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const int bn = M <= 32 ? 32 : M <= 64 ? 64 : 128;
    CUtensorMap maps[4];
    if (!encode_u32_map(&maps[2], xh, M, K, kTK, bn, true) || !encode_u32_map(&maps[3], xl, M, K, kTK, bn, true))
        return cudaErrorInvalidValue;
    for (int64_t n0 = 0; n0 < N; n0 += rows) {
        const int64_t rr = std::min(rows, N - n0);
        const uint8_t* ws = W + n0 * nb * kBlockBytes;  // the slice's first block
        if (type == kTypePn3t)
            launch_decode_slice<kTypePn3t>(ws, rr * nb, wh, wl, sms, stream);
        else
            launch_decode_slice<kTypePn4t>(ws, rr * nb, wh, wl, sms, stream);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        if (!encode_u32_map(&maps[0], wh, rr, K, kTK, kTM, true) || !encode_u32_map(&maps[1], wl, rr, K, kTK, kTM, true))
            return cudaErrorInvalidValue;
        GemmArgs a{};
        a.Y = Y;
        a.err = err;
        a.M = static_cast<int>(M);
        a.rows = static_cast<int>(rr);
        a.K = static_cast<int>(K);
        a.ldy = N;
        a.n0 = n0;
        // K split over a cluster while the slice's tiles would fill fewer SMs than they could
        // (every share keeps at least 8 K tiles)
        {
            const int64_t tiles = (rr + kTM - 1) / kTM * ((M + bn - 1) / bn);
            const int64_t nk = (K + kTK - 1) / kTK;
            a.ks = 1;
            while (a.ks < 8 && tiles * (a.ks + 1) <= sms && nk >= 8 * (a.ks + 1)) ++a.ks;
        }
        e = (bn == 32) ? launch_gemm_bn<32>(maps, a, stream)
            : (bn == 64) ? launch_gemm_bn<64>(maps, a, stream)
                         : launch_gemm_bn<128>(maps, a, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace pnq
