// pnq_internal.h -- host-side launchers shared by the translation units of libpnq.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace pnq {

struct Nvfp4View {
    const uint8_t* codes;   // device [N][K/2], low nibble = even k
    const uint8_t* scales;  // device [N][K/16] E4M3FN
    float g;                // global multiplier
};

// Configuration of the tensor-core GEMV (fast path); fields <= 0 are chosen automatically.
struct MmaConfig {
    int tpw;   // row tiles of 16 per consumer warp (1: 16 consumer warps, 2: 8)
    int grid;  // CTAs (at most one per SM)
    int rb;    // operand ring slots
    int ns;    // weight pipeline stages
    int order; // wide batches: 1 = tile-major items with streamed operands, 2 = grouped unit-major
               // items with resident operands
    int pf;    // static weights: stages requested before the previous grid completes (0 = all)
};

// Workspace handed in by the caller (nullptr ws: the per-stream workspace is used).
struct ExtWorkspace {
    float* ws = nullptr;
    uint32_t* cnt = nullptr;
    size_t floats = 0, counters = 0;
};

int device_sm_count();

// 2-D tensor map over a row-major u32 matrix [rows][row_u32] (row pitch a multiple of 16
// bytes) with box {box_x, box_y}; rows past the end read as zeros. swizzle_128b: the copy
// stores 16-byte chunk c of box row r at chunk c ^ (r % 8) of that row (box rows of 128 bytes,
// shared destination 1024-byte aligned). False when the driver entry point is missing or the
// encoder rejects the arguments.
bool encode_u32_map(CUtensorMap* map, const void* base, int64_t rows, int64_t row_u32, int box_x, int box_y,
                    bool swizzle_128b = false);

// Workspace of the stream-K GEMV kernels, one per (device, stream): `floats` partial sums and
// `counters` tile counters (zero between launches). Grows on demand; outgrown buffers stay
// allocated because a captured graph may still refer to them. Allocation is allowed while the
// stream is being captured (the counters are then cleared by a captured memset node).
cudaError_t stream_workspace(cudaStream_t stream, size_t floats, size_t counters, float** ws, uint32_t** cnt);

cudaError_t launch_pn_dequant(int type, const uint8_t* W, int64_t n_rows, int64_t K, float* out,
                              cudaStream_t stream);
cudaError_t launch_nvfp4_dequant(const Nvfp4View& w, int64_t n_rows, int64_t K, float* out,
                                 cudaStream_t stream);
cudaError_t launch_pn_validate(int type, const uint8_t* W, int64_t n_rows, int64_t K, int32_t* flags,
                               cudaStream_t stream);
cudaError_t launch_nvfp4_validate(const Nvfp4View& w, int64_t n_rows, int64_t K, int32_t* flags,
                                  cudaStream_t stream);

// Generic path: any 2-byte aligned PN buffer / any NVFP4 layout, CUDA-core FMA.
cudaError_t launch_pn_gemv_simt(int type, const uint8_t* W, int64_t N, int64_t K, const float* X, int M,
                                float* Y, cudaStream_t stream);
cudaError_t launch_nvfp4_gemv_simt(const Nvfp4View& w, int64_t N, int64_t K, const uint16_t* X, int M,
                                   float* Y, cudaStream_t stream);

// Fast path: 16-byte aligned weights and x, bulk-copy pipeline, mma.sync decode-and-multiply.
// static_weights: the weights are not written by work queued earlier in the stream, so they
// may be prefetched before the previous grid completes. Returns cudaErrorNotSupported when
// the shape is outside the fast path's range (the caller then uses the generic path).
cudaError_t launch_pn_gemv_mma(int type, const uint8_t* W, int64_t N, int64_t K, const float* X, int M,
                               float* Y, int* err, MmaConfig cfg, bool static_weights, cudaStream_t stream,
                               const ExtWorkspace& ext = ExtWorkspace{});
// Tensor-core path (tcgen05, tensor memory): 16-byte aligned weights and x, (K / block) a
// multiple of 8. Keeps a per-(device, stream) workspace of partial rows. Returns
// cudaErrorNotSupported outside its range.
cudaError_t launch_pn_gemv_tc(int type, const uint8_t* W, int64_t N, int64_t K, const float* X, int M, float* Y,
                              int* err, bool static_weights, cudaStream_t stream);
cudaError_t launch_nvfp4_gemv_mma(const Nvfp4View& w, int64_t N, int64_t K, const uint16_t* X, int M,
                                  float* Y, int* err, MmaConfig cfg, bool static_weights, cudaStream_t stream,
                                  const ExtWorkspace& ext = ExtWorkspace{});

}  // namespace pnq
