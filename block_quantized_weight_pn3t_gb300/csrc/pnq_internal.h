// pnq_internal.h -- host-side launchers shared by the translation units of libpnq.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace pnq {

struct Nvfp4View {
    const uint8_t* codes;   // device [N][K/2], low nibble = even k
    const uint8_t* scales;  // device [N][K/16] E4M3FN
    float g;                // global multiplier (div: the global divisor d_w)
    bool div = false;       // the weight is e2m1 * e4m3 / g
};

// Planes of a grouped signed-integer matrix (pnq_grouped.cu states the layout).
struct GroupedView {
    const uint8_t* lo;
    const uint8_t* hi;
    const uint16_t* scales;
};
struct GroupedOut {
    uint8_t* lo;
    uint8_t* hi;
    uint16_t* scales;
};

int device_sm_count();

// 2-D tensor map over a row-major u32 matrix [rows][row_u32] (row pitch a multiple of 16
// bytes) with box {box_x, box_y}; rows past the end read as zeros. swizzle_128b: the copy
// stores 16-byte chunk c of box row r at chunk c ^ (r % 8) of that row (box rows of 128 bytes,
// shared destination 1024-byte aligned). False when the driver entry point is missing or the
// encoder rejects the arguments.
bool encode_u32_map(CUtensorMap* map, const void* base, int64_t rows, int64_t row_u32, int box_x, int box_y,
                    bool swizzle_128b = false);

cudaError_t launch_pn_dequant(int type, const uint8_t* W, int64_t n_rows, int64_t K, float* out,
                              cudaStream_t stream);
cudaError_t launch_nvfp4_dequant(const Nvfp4View& w, int64_t n_rows, int64_t K, float* out,
                                 cudaStream_t stream);
cudaError_t launch_pn_validate(int type, const uint8_t* W, int64_t n_rows, int64_t K, int32_t* flags,
                               cudaStream_t stream);
cudaError_t launch_nvfp4_validate(const Nvfp4View& w, int64_t n_rows, int64_t K, int32_t* flags,
                                  cudaStream_t stream);

// Grouped signed-integer formats (type = kTypeQ4G64 ..): bit-exact dequantize, validate, GEMV on
// the CUDA cores (X fp32), and the canonical encoder MAXABS_F16_RECIP_RNE_V1 (status[r] = 1 for
// a row with a non-finite weight or a scale that overflows binary16; zeroed first).
cudaError_t launch_grouped_dequant(int type, const GroupedView& v, int64_t n_rows, int64_t K, float* out,
                                   cudaStream_t stream);
cudaError_t launch_grouped_validate(int type, const GroupedView& v, int64_t n_rows, int64_t K, int32_t* flags,
                                    cudaStream_t stream);
cudaError_t launch_grouped_gemv(int type, const GroupedView& v, int64_t N, int64_t K, const float* X, int M,
                                float* Y, cudaStream_t stream);
cudaError_t launch_grouped_quantize(int type, const float* w, int64_t n_rows, int64_t K, const GroupedOut& out,
                                    int32_t* status, cudaStream_t stream);

// PN reference quantizer, bit-exact with the CPU reference (status[r] = 1 for a row with a
// non-finite weight; zeroed first).
cudaError_t launch_pn_quantize(int type, const float* w, int64_t n_rows, int64_t K, uint8_t* out, int32_t* status,
                               cudaStream_t stream);

// NVFP4 clip search (TandemLLM "Quantisation and profiles"), bit-exact with the CPU reference;
// status[r] = 1 for a row with a non-finite weight (zeroed first).
cudaError_t launch_nvfp4_clip(const float* w, const float* act_ms, float g, int64_t n_rows, int64_t K, uint8_t* codes,
                              uint8_t* scales, int32_t* status, cudaStream_t stream);

// PN products for any M on the tcgen05 tensor cores (prefill): x split into two tf32 planes, the
// weights decoded slice by slice into two tf32 planes, three tf32 MMAs per K step (pnq_prefill.cu).
// scratch: 8 * M * K bytes for x plus 8 * K bytes per weight row of a slice (slices of a multiple
// of 128 rows); cudaErrorMemoryAllocation when it holds less than one 128-row slice.
int64_t prefill_slice_rows(int64_t N, int64_t K, int64_t M, size_t scratch_bytes);
cudaError_t launch_pn_prefill(int type, const uint8_t* W, int64_t N, int64_t K, const float* X, int64_t M, float* Y,
                              int* err, void* scratch, size_t scratch_bytes, cudaStream_t stream);

// Generic path: any 2-byte aligned PN buffer / any NVFP4 layout, CUDA-core FMA.
cudaError_t launch_pn_gemv_simt(int type, const uint8_t* W, int64_t N, int64_t K, const float* X, int M,
                                float* Y, cudaStream_t stream);
cudaError_t launch_nvfp4_gemv_simt(const Nvfp4View& w, int64_t N, int64_t K, const uint16_t* X, int M,
                                   float* Y, cudaStream_t stream);

// Fast path: 16-byte aligned weights and x, (K / block) a multiple of 8; clusters of one or two
// CTAs own disjoint row ranges and sum their partials on chip (no workspace). static_weights: the
// weights are not written by work queued earlier in the stream, so they may be streamed before
// the previous grid completes. cluster / stages > 0 force the plan (tests); 0 = automatic.
// Returns cudaErrorNotSupported when the shape is outside the fast path's range (the caller then
// uses the generic path).
cudaError_t launch_pn_gemv_mma(int type, const uint8_t* W, int64_t N, int64_t K, const float* X, int M,
                               float* Y, int* err, int cluster, int stages, bool static_weights,
                               cudaStream_t stream);
// Same pipeline for NVFP4: codes, scales and x 16-byte aligned, K % 256 == 0.
cudaError_t launch_nvfp4_gemv_mma(const Nvfp4View& w, int64_t N, int64_t K, const uint16_t* X, int M,
                                  float* Y, int* err, int cluster, int stages, bool static_weights,
                                  cudaStream_t stream);

}  // namespace pnq
