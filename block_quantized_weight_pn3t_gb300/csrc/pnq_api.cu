// pnq_api.cu -- the C ABI declared in include/pnq.h: argument checks, kernel choice, status codes.
#include "pnq.h"
#include "pnq_device.cuh"
#include "pnq_internal.h"

#include <algorithm>
#include <atomic>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

// Device error word: 0, or the site code of the first bounded wait that gave up (one copy per
// device that loads the library).
__device__ int g_pnq_error_word = 0;

namespace pnq {

namespace {

constexpr int kMaxDevices = 64;

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

// Device address of a library __device__ symbol on the current device, looked up once per
// device (host threads may race on the first lookup; they store the same address).
template <typename T>
T* symbol_address(std::atomic<T*> (&cache)[kMaxDevices], const void* symbol) {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    T* p = cache[dev].load(std::memory_order_relaxed);
    if (!p) {
        void* q = nullptr;
        if (cudaGetSymbolAddress(&q, symbol) != cudaSuccess) return nullptr;
        p = static_cast<T*>(q);
        cache[dev].store(p, std::memory_order_relaxed);
    }
    return p;
}

std::atomic<int*> g_error_word_ptrs[kMaxDevices];

int* error_word() { return symbol_address(g_error_word_ptrs, static_cast<const void*>(&g_pnq_error_word)); }

// "auto" (default: the mma.sync path whenever eligible), "simt" (generic path only) or "mma"
// (same as auto).
int forced_kernel() {
    static int mode = [] {
        const char* s = std::getenv("PNQ_FORCE_KERNEL");
        if (s && std::strcmp(s, "simt") == 0) return 1;
        if (s && std::strcmp(s, "mma") == 0) return 2;
        return 0;
    }();
    return mode;
}

int block_weights(int type) {
    if (type == PNQ_PN3T) return 80;
    if (type == PNQ_PN4T) return 64;
    return 0;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int map_cuda(cudaError_t e) { return e == cudaSuccess ? PNQ_OK : PNQ_ERR_CUDA; }

bool is_grouped(int type) {
    return type == PNQ_Q4G64_F16S || type == PNQ_Q5G64_F16S || type == PNQ_Q6G64_F16S || type == PNQ_W8G32_F16S;
}

int grouped_bits(int type) {
    return type == PNQ_Q4G64_F16S ? 4 : type == PNQ_Q5G64_F16S ? 5 : type == PNQ_Q6G64_F16S ? 6 : 8;
}

// Grouped planes: K % 8 == 0 (whole octets per row), the planes present and aligned for the
// kernels' loads (row strides keep the base alignment because K % 8 == 0).
int check_grouped_planes(int type, int64_t rows, const uint8_t* lo, const uint8_t* hi, const uint16_t* scales) {
    const int bits = grouped_bits(type);
    if (rows > 0 && (!lo || !scales || ((bits == 5 || bits == 6) && !hi))) return PNQ_ERR_NULL;
    if (!aligned(lo, bits == 8 ? 8 : 4) || !aligned(scales, 2) || (bits == 6 && !aligned(hi, 2)))
        return PNQ_ERR_ALIGN;
    return PNQ_OK;
}

int check_grouped(int type, const void* W, int64_t rows, int64_t K, GroupedView* v) {
    if (rows < 0 || K <= 0 || K % 8 != 0 || rows > INT64_MAX / K) return PNQ_ERR_SHAPE;
    if (!W) return PNQ_ERR_NULL;
    const pnq_grouped_weights* d = static_cast<const pnq_grouped_weights*>(W);
    v->lo = d->lo;
    v->hi = d->hi;
    v->scales = d->scales;
    return check_grouped_planes(type, rows, d->lo, d->hi, d->scales);
}

// Shared shape / pointer checks. On success fills the NVFP4 view (when type is NVFP4).
int check_common(int type, const void* W, int64_t rows, int64_t K, Nvfp4View* nv) {
    if (type != PNQ_PN3T && type != PNQ_PN4T && type != PNQ_NVFP4 && type != PNQ_NVFP4_DIV) return PNQ_ERR_TYPE;
    if (rows < 0 || K <= 0) return PNQ_ERR_SHAPE;
    if (type == PNQ_NVFP4 || type == PNQ_NVFP4_DIV) {
        if (K % 16 != 0) return PNQ_ERR_SHAPE;
        if (rows > INT64_MAX / K) return PNQ_ERR_SHAPE;
        if (!W) return PNQ_ERR_NULL;
        const pnq_nvfp4_weights* d = static_cast<const pnq_nvfp4_weights*>(W);
        if (rows > 0 && (!d->codes || !d->scales)) return PNQ_ERR_NULL;
        nv->codes = d->codes;
        nv->scales = d->scales;
        nv->g = d->global_scale;
        nv->div = type == PNQ_NVFP4_DIV;
        return PNQ_OK;
    }
    const int blk = block_weights(type);
    if (K % blk != 0) return PNQ_ERR_SHAPE;
    if (rows > INT64_MAX / (K / blk * 34) || rows > INT64_MAX / K) return PNQ_ERR_SHAPE;
    if (rows > 0 && !W) return PNQ_ERR_NULL;
    if (!aligned(W, 2)) return PNQ_ERR_ALIGN;
    return PNQ_OK;
}

}  // namespace

int device_sm_count() {
    static std::atomic<int> counts[kMaxDevices];
    const int dev = current_device();
    if (dev < 0) return 148;
    int n = counts[dev].load(std::memory_order_relaxed);
    if (!n) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        counts[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

namespace {

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn tensor_map_encoder() {
    static EncodeFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeFn>(nullptr);
        return reinterpret_cast<EncodeFn>(p);
    }();
    return fn;
}

}  // namespace

bool encode_u32_map(CUtensorMap* map, const void* base, int64_t rows, int64_t row_u32, int box_x, int box_y,
                    bool swizzle_128b) {
    EncodeFn enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_u32), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_u32 * 4)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_x), static_cast<cuuint32_t>(box_y)};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_128b ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace pnq

using namespace pnq;

namespace {

int gemv_impl(int type, const void* W, int64_t N, int64_t K, const void* X, int M, float* Y, unsigned int flags,
              cudaStream_t stream) {
    if (is_grouped(type)) {
        GroupedView v{};
        const int rc = check_grouped(type, W, N, K, &v);
        if (rc != PNQ_OK) return rc;
        if (M < 1 || M > 16 || static_cast<int64_t>(M) > INT64_MAX / K) return PNQ_ERR_SHAPE;
        if ((flags & ~static_cast<unsigned int>(PNQ_GEMV_STATIC_WEIGHTS)) != 0) return PNQ_ERR_FLAGS;
        if (N == 0) return PNQ_OK;
        if (!X || !Y) return PNQ_ERR_NULL;
        if (!aligned(X, 16) || !aligned(Y, 4)) return PNQ_ERR_ALIGN;
        return map_cuda(launch_grouped_gemv(type, v, N, K, static_cast<const float*>(X), M, Y, stream));
    }
    Nvfp4View nv{};
    int rc = check_common(type, W, N, K, &nv);
    if (rc != PNQ_OK) return rc;
    if (M < 1 || M > 16) return PNQ_ERR_SHAPE;
    if (static_cast<int64_t>(M) > INT64_MAX / K) return PNQ_ERR_SHAPE;
    if ((flags & ~static_cast<unsigned int>(PNQ_GEMV_STATIC_WEIGHTS)) != 0) return PNQ_ERR_FLAGS;
    if (N == 0) return PNQ_OK;
    if (!X || !Y) return PNQ_ERR_NULL;
    if (!aligned(Y, 4)) return PNQ_ERR_ALIGN;
    const bool static_w = (flags & PNQ_GEMV_STATIC_WEIGHTS) != 0;
    const int mode = forced_kernel();
    if (type == PNQ_NVFP4 || type == PNQ_NVFP4_DIV) {
        if (!aligned(X, 2)) return PNQ_ERR_ALIGN;
        const uint16_t* x = static_cast<const uint16_t*>(X);
        // the fast path scales by a multiplier: for a divisor d_w, fp32(1 / d_w) when that is a
        // normal number (a relative change of at most 2^-24 per weight, inside the accuracy
        // bound); otherwise the generic path divides each output by d_w
        Nvfp4View fast = nv;
        if (nv.div) {
            fast.g = 1.0f / nv.g;
            fast.div = false;
        }
        const bool mult_ok = !nv.div || (fast.g >= 1.17549435e-38f && fast.g <= 3.4028234663852886e38f);
        if (mode != 1 && mult_ok && aligned(nv.codes, 16) && aligned(nv.scales, 16) && aligned(x, 16) &&
            K % 256 == 0) {
            const cudaError_t e = launch_nvfp4_gemv_mma(fast, N, K, x, M, Y, error_word(), 0, 0, static_w, stream);
            if (e != cudaErrorNotSupported) return map_cuda(e);
        }
        return map_cuda(launch_nvfp4_gemv_simt(nv, N, K, x, M, Y, stream));
    }
    if (!aligned(X, 4)) return PNQ_ERR_ALIGN;
    const uint8_t* w = static_cast<const uint8_t*>(W);
    const float* x = static_cast<const float*>(X);
    if (mode != 1 && aligned(w, 16) && (K / block_weights(type)) % 8 == 0) {
        const cudaError_t e = launch_pn_gemv_mma(type, w, N, K, x, M, Y, error_word(), 0, 0, static_w, stream);
        if (e != cudaErrorNotSupported) return map_cuda(e);
    }
    return map_cuda(launch_pn_gemv_simt(type, w, N, K, x, M, Y, stream));
}

}  // namespace

extern "C" int pnq_gemv_ex(int type, const void* W, int64_t N, int64_t K, const void* X, int M, float* Y,
                           unsigned int flags, cudaStream_t stream) {
    return gemv_impl(type, W, N, K, X, M, Y, flags, stream);
}

extern "C" int pnq_gemv_noalloc(int type, const void* W, int64_t N, int64_t K, const void* X, int M, float* Y,
                                unsigned int flags, cudaStream_t stream) {
    return gemv_impl(type, W, N, K, X, M, Y, flags, stream);
}

extern "C" int pnq_gemm_scratch_bytes(int type, int64_t N, int64_t K, int64_t M, int64_t slice_rows,
                                      uint64_t* bytes) {
    if (type != PNQ_PN3T && type != PNQ_PN4T) return PNQ_ERR_TYPE;
    if (!bytes) return PNQ_ERR_NULL;
    const int blk = block_weights(type);
    if (N < 0 || K <= 0 || K % blk != 0 || M < 1 || slice_rows < 0) return PNQ_ERR_SHAPE;
    int64_t rows = slice_rows > 0 ? slice_rows : N;
    rows = (rows + 127) / 128 * 128;
    if (rows == 0) rows = 128;
    if (M > INT64_MAX / 8 / K || rows > INT64_MAX / 8 / K - M) return PNQ_ERR_SHAPE;
    *bytes = static_cast<uint64_t>(8 * K * (M + rows));
    return PNQ_OK;
}

extern "C" int pnq_gemm(int type, const void* W, int64_t N, int64_t K, const float* X, int64_t M, float* Y,
                        void* scratch, uint64_t scratch_bytes, cudaStream_t stream) {
    if (type != PNQ_PN3T && type != PNQ_PN4T) return PNQ_ERR_TYPE;
    Nvfp4View nv{};
    const int rc = check_common(type, W, N, K, &nv);
    if (rc != PNQ_OK) return rc;
    if (M < 1 || M > INT32_MAX / 2 || K > INT32_MAX || N > INT32_MAX || M > INT64_MAX / 8 / K) return PNQ_ERR_SHAPE;
    if (N == 0) return PNQ_OK;
    if (!X || !Y || !scratch) return PNQ_ERR_NULL;
    if (!aligned(X, 16) || !aligned(Y, 4) || !aligned(scratch, 16)) return PNQ_ERR_ALIGN;
    if (prefill_slice_rows(N, K, M, static_cast<size_t>(scratch_bytes)) < 128) return PNQ_ERR_SCRATCH;
    return map_cuda(launch_pn_prefill(type, static_cast<const uint8_t*>(W), N, K, X, M, Y, error_word(), scratch,
                                      static_cast<size_t>(scratch_bytes), stream));
}

extern "C" int pnq_gemv(int type, const void* W, int64_t N, int64_t K, const void* X, int M, float* Y,
                        cudaStream_t stream) {
    return pnq_gemv_ex(type, W, N, K, X, M, Y, 0u, stream);
}

extern "C" int pnq_dequantize_row(int type, const void* W, int64_t n_rows, int64_t K, float* out,
                                  cudaStream_t stream) {
    if (is_grouped(type)) {
        GroupedView v{};
        const int rc = check_grouped(type, W, n_rows, K, &v);
        if (rc != PNQ_OK) return rc;
        if (n_rows == 0) return PNQ_OK;
        if (!out) return PNQ_ERR_NULL;
        if (!aligned(out, 16)) return PNQ_ERR_ALIGN;
        return map_cuda(launch_grouped_dequant(type, v, n_rows, K, out, stream));
    }
    Nvfp4View nv{};
    int rc = check_common(type, W, n_rows, K, &nv);
    if (rc != PNQ_OK) return rc;
    if (n_rows == 0) return PNQ_OK;
    if (!out) return PNQ_ERR_NULL;
    if (!aligned(out, 4)) return PNQ_ERR_ALIGN;
    if (type == PNQ_NVFP4 || type == PNQ_NVFP4_DIV) return map_cuda(launch_nvfp4_dequant(nv, n_rows, K, out, stream));
    return map_cuda(launch_pn_dequant(type, static_cast<const uint8_t*>(W), n_rows, K, out, stream));
}

extern "C" int pnq_validate_row(int type, const void* W, int64_t n_rows, int64_t K, int32_t* flags,
                                cudaStream_t stream) {
    if (is_grouped(type)) {
        GroupedView v{};
        const int rc = check_grouped(type, W, n_rows, K, &v);
        if (rc != PNQ_OK) return rc;
        if (n_rows == 0) return PNQ_OK;
        if (!flags) return PNQ_ERR_NULL;
        if (!aligned(flags, 4)) return PNQ_ERR_ALIGN;
        return map_cuda(launch_grouped_validate(type, v, n_rows, K, flags, stream));
    }
    Nvfp4View nv{};
    int rc = check_common(type, W, n_rows, K, &nv);
    if (rc != PNQ_OK) return rc;
    if (n_rows == 0) return PNQ_OK;
    if (!flags) return PNQ_ERR_NULL;
    if (!aligned(flags, 4)) return PNQ_ERR_ALIGN;
    if (type == PNQ_NVFP4 || type == PNQ_NVFP4_DIV) return map_cuda(launch_nvfp4_validate(nv, n_rows, K, flags, stream));
    return map_cuda(launch_pn_validate(type, static_cast<const uint8_t*>(W), n_rows, K, flags, stream));
}

extern "C" int pnq_quantize_row(int type, const float* w, int64_t n_rows, int64_t K, void* out, int32_t* row_status,
                                cudaStream_t stream) {
    if (type != PNQ_PN3T && type != PNQ_PN4T && !is_grouped(type)) return PNQ_ERR_TYPE;
    if (n_rows < 0 || K <= 0 || n_rows > INT64_MAX / K) return PNQ_ERR_SHAPE;
    if (is_grouped(type)) {
        if (K % 8 != 0) return PNQ_ERR_SHAPE;
        if (!out) return PNQ_ERR_NULL;
        const pnq_grouped_planes* p = static_cast<const pnq_grouped_planes*>(out);
        int rc = check_grouped_planes(type, n_rows, p->lo, p->hi, p->scales);
        if (rc != PNQ_OK) return rc;
        if (n_rows == 0) return PNQ_OK;
        if (!w || !row_status) return PNQ_ERR_NULL;
        if (!aligned(w, 4) || !aligned(row_status, 4)) return PNQ_ERR_ALIGN;
        return map_cuda(launch_grouped_quantize(type, w, n_rows, K, GroupedOut{p->lo, p->hi, p->scales}, row_status,
                                                stream));
    }
    const int blk = block_weights(type);
    if (K % blk != 0 || n_rows > INT64_MAX / (K / blk * 34)) return PNQ_ERR_SHAPE;
    if (n_rows == 0) return PNQ_OK;
    if (!w || !out || !row_status) return PNQ_ERR_NULL;
    if (!aligned(w, 4) || !aligned(out, 2) || !aligned(row_status, 4)) return PNQ_ERR_ALIGN;
    return map_cuda(launch_pn_quantize(type, w, n_rows, K, static_cast<uint8_t*>(out), row_status, stream));
}

extern "C" int pnq_quantize_nvfp4_clip(const float* w, const float* act_ms, int64_t n_rows, int64_t K,
                                       float global_scale, uint8_t* codes, uint8_t* scales, int32_t* row_status,
                                       cudaStream_t stream) {
    if (n_rows < 0 || K <= 0 || K % 16 != 0 || n_rows > INT64_MAX / K) return PNQ_ERR_SHAPE;
    if (!(global_scale > 0.0f && global_scale <= 3.4028234663852886e38f)) return PNQ_ERR_VALUE;
    if (n_rows == 0) return PNQ_OK;
    if (!w || !act_ms || !codes || !scales || !row_status) return PNQ_ERR_NULL;
    if (!aligned(w, 4) || !aligned(act_ms, 4) || !aligned(row_status, 4)) return PNQ_ERR_ALIGN;
    return map_cuda(launch_nvfp4_clip(w, act_ms, global_scale, n_rows, K, codes, scales, row_status, stream));
}

namespace pnq {

// One thread waits, bounded by limit_ns, on a shared-memory barrier nothing arrives at, with the
// kernels' own bounded wait, and records the self-test site code when the wait runs out.
__global__ void wait_selftest_kernel(int* err, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&bar), 1);
        mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait_bounded(smem_addr(&bar), 0, limit_ns)) record_error(err, kErrSelfTest);
}

}  // namespace pnq

extern "C" int pnq_selftest_wait(uint32_t limit_us, cudaStream_t stream) {
    if (limit_us == 0 || limit_us > 2000000u) return PNQ_ERR_VALUE;
    int* err = error_word();
    if (!err) return PNQ_ERR_CUDA;
    wait_selftest_kernel<<<1, 32, 0, stream>>>(err, static_cast<uint64_t>(limit_us) * 1000ull);
    return map_cuda(cudaGetLastError());
}

extern "C" int pnq_device_error(int32_t* code) {
    if (!code) return PNQ_ERR_NULL;
    int v = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return PNQ_ERR_CUDA;  // every stream, not only the default one
    if (cudaMemcpyFromSymbol(&v, g_pnq_error_word, sizeof(int)) != cudaSuccess) return PNQ_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_pnq_error_word, &zero, sizeof(int)) != cudaSuccess) return PNQ_ERR_CUDA;
    *code = v;
    return v == 0 ? PNQ_OK : PNQ_ERR_DEVICE;
}

extern "C" const char* pnq_version(void) { return "pnq 0.1.0 (sm_103a)"; }
