/*
 * pnq_oracle.h -- CPU oracle for the PN weight formats (pn3t, pn4t) and NVFP4.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT. Only the test suite, the smoke
 * check and the benchmark's CPU-baseline / reference legs may load this. The
 * CUDA library shares no code, header, table or constant with it.
 *
 * Every routine is a plain, slow restatement of a definition on the source pages:
 *   - "PN weight format" (tensorless docs, reference/pn-format): Types, Block layout,
 *     Value, Reference quantizer, Validation, "Where PN runs".
 *   - NInfer "tensor-formats.md": section 3.1 (BF16), section 3.3 (NVFP4, E2M1, E4M3FN).
 *   - TandemLLM "Quantisation and profiles", section NVFP4: weight =
 *     e2m1(code) * weight_scale[n, k // 16] * weight_scale_2 (global multiplier).
 * Floating point is fp64 unless the page fixes another precision.
 *
 * Parity status: every function here is pinned by tests/test_oracle_*.py except
 * pnq_ref_quantize_row, whose bitwise agreement with the engine's own quantizer
 * is "parity unpinned" (the engine's golden test file is not available); the
 * quantizer is pinned only by invariants, exhaustive re-scoring and tie cases.
 */
#ifndef PNQ_ORACLE_H
#define PNQ_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { PNQ_REF_PN3T = 124, PNQ_REF_PN4T = 125, PNQ_REF_NVFP4 = 1004 };
/* grouped signed-integer formats ("tensor-formats.md" sections 4-7; the ids are this library's) */
enum { PNQ_REF_Q4G64 = 1104, PNQ_REF_Q5G64 = 1105, PNQ_REF_Q6G64 = 1106, PNQ_REF_W8G32 = 1108 };
enum { PNQ_REF_OK = 0, PNQ_REF_ERR_TYPE = -1, PNQ_REF_ERR_SHAPE = -2,
       PNQ_REF_ERR_NULL = -3, PNQ_REF_ERR_VALUE = -6 };

/* Weights per 34-byte block (80 for pn3t, 64 for pn4t), 0 for other types. */
int pnq_ref_block_weights(int type);

/* Scalar codecs, written from the bit definitions. */
double   pnq_ref_fp16_to_double(uint16_t h);
uint16_t pnq_ref_double_to_fp16(double x);          /* one round-to-nearest-even step */
double   pnq_ref_bf16_to_double(uint16_t b);
double   pnq_ref_e2m1_to_double(uint8_t c);          /* low 4 bits used */
double   pnq_ref_e4m3fn_to_double(uint8_t c);

/* PN rows: W = n_rows * (K / BLK) blocks of 34 bytes, row-major. out: fp32 [n_rows][K]. */
int pnq_ref_dequantize_row(int type, const uint8_t* W, int64_t n_rows, int64_t K, float* out);
/* Negative control: the documented wrong CPU decode (shift by element index). */
int pnq_ref_dequantize_row_elemshift(int type, const uint8_t* W, int64_t n_rows, int64_t K, float* out);
/* flags[r] = 1 if row r is invalid, else 0. */
int pnq_ref_validate_row(int type, const uint8_t* W, int64_t n_rows, int64_t K, int32_t* flags);
/* Reference quantizer: K fp32 weights of one row -> K/BLK blocks. chosen_m (nullable)
 * receives the chosen multiplier per block (0 for the canonical zero group). */
int pnq_ref_quantize_row(int type, const float* w, int64_t K, uint8_t* out, double* chosen_m);

/* NVFP4: codes [n_rows][K/2] (low nibble = even k), scales [n_rows][K/16] E4M3FN,
 * g = fp32 global multiplier. */
int pnq_ref_dequantize_row_nvfp4(const uint8_t* codes, const uint8_t* scales, float g,
                                 int64_t n_rows, int64_t K, float* out);
int pnq_ref_validate_row_nvfp4(const uint8_t* scales, float g, int64_t n_rows, int64_t K,
                               int32_t* flags);

/* GEMV: Y[m][n] = sum_k w[n][k] * x[m][k] in fp64, A[m][n] = sum_k |w[n][k] * x[m][k]|.
 * PN takes fp32 X [M][K]; NVFP4 takes bf16 X [M][K] (raw 16-bit words).
 * Y and A are fp64 [M][N]; A may be NULL. */
int pnq_ref_gemv(int type, const uint8_t* W, int64_t N, int64_t K, const float* X, int M,
                 double* Y, double* A);
/* NVFP4 with the global field read as a divisor d_w ("tensor-formats.md" section 3.3):
 * out = fp32(e2m1 * e4m3) / d_w (one rounding); the GEMV divides the exact product in fp64. */
int pnq_ref_dequantize_row_nvfp4_div(const uint8_t* codes, const uint8_t* scales, float dw,
                                     int64_t n_rows, int64_t K, float* out);
int pnq_ref_gemv_nvfp4_div(const uint8_t* codes, const uint8_t* scales, float dw, int64_t N,
                           int64_t K, const uint16_t* X, int M, double* Y, double* A);
int pnq_ref_gemv_nvfp4(const uint8_t* codes, const uint8_t* scales, float g, int64_t N,
                       int64_t K, const uint16_t* X, int M, double* Y, double* A);

/* Grouped signed-integer formats ("tensor-formats.md" sections 4 to 7), in the library's plane
 * layout (pnq_oracle.c states it): plane sizes per row, decode, validity, the canonical encoder
 * MAXABS_F16_RECIP_RNE_V1 (section 7) and the GEMV over the reconstructed binary32 weights. */
int pnq_ref_grouped_plane_bytes(int type, int64_t K, int64_t* lo_bytes, int64_t* hi_bytes, int64_t* n_scales);
int pnq_ref_dequantize_grouped(int type, const uint8_t* lo, const uint8_t* hi, const uint16_t* sc,
                               int64_t n_rows, int64_t K, float* out);
int pnq_ref_validate_grouped(int type, const uint8_t* lo, const uint8_t* hi, const uint16_t* sc,
                             int64_t n_rows, int64_t K, int32_t* flags);
int pnq_ref_quantize_grouped(int type, const float* w, int64_t n_rows, int64_t K, uint8_t* lo,
                             uint8_t* hi, uint16_t* sc, int64_t* fail_row);
int pnq_ref_gemv_grouped(int type, const uint8_t* lo, const uint8_t* hi, const uint16_t* sc, int64_t N,
                         int64_t K, const float* X, int M, double* Y, double* A);

/* NVFP4 clip search (TandemLLM "Quantisation and profiles", section "The clip search"): per group
 * of 16, the multiplier of 1.00, 0.95, 0.90, 0.85, 0.80 on the base scale amax / (6 g) with the
 * least act_ms-weighted squared error; codes [N][K/2], scales [N][K/16] E4M3FN; chosen (may be
 * NULL) receives the index of the multiplier kept per group. pnq_oracle.c states the readings. */
int pnq_ref_quantize_nvfp4_clip(const float* w, const float* act_ms, float g, int64_t n_rows, int64_t K,
                                uint8_t* codes, uint8_t* scales, int32_t* chosen);

#ifdef __cplusplus
}
#endif
#endif
