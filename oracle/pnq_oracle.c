/*
 * pnq_oracle.c -- CPU oracle for pn3t / pn4t / NVFP4.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT: only the test suite, the smoke
 * check and the benchmark's CPU-baseline / reference legs load this library.
 * It is deliberately slow and literal: no blocking, no vectorisation, no fused
 * steps. Every routine cites the passage of the source pages it restates.
 * Parity of pnq_ref_quantize_row against the engine's own quantizer is
 * "parity unpinned" (no printed worked example exists); see pnq_oracle.h.
 */
#include "pnq_oracle.h"

#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

/* ---- format constants ("PN weight format", section Types) ------------------ */

typedef struct {
    int blk;   /* weights per block */
    int bits;  /* bits per code */
    int cpw;   /* codes per u32 word */
    int z;     /* zero point 2^(bits-1) */
} pn_params;

static int pn_lookup(int type, pn_params* p) {
    if (type == PNQ_REF_PN3T) { p->blk = 80; p->bits = 3; p->cpw = 10; p->z = 4; return 1; }
    if (type == PNQ_REF_PN4T) { p->blk = 64; p->bits = 4; p->cpw = 8;  p->z = 8; return 1; }
    return 0;
}

int pnq_ref_block_weights(int type) {
    pn_params p;
    return pn_lookup(type, &p) ? p.blk : 0;
}

/* ---- scalar codecs ------------------------------------------------------- */

/* IEEE-754 binary16: sign bit 15, 5-bit exponent (bias 15), 10-bit fraction. */
double pnq_ref_fp16_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* zero or subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp(1024.0 + (double)f, e - 25);     /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* One round-to-nearest-even step from fp64 to binary16; overflow gives infinity. */
uint16_t pnq_ref_double_to_fp16(double x) {
    if (isnan(x)) return 0x7E00;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0) return sign;
    if (isinf(a)) return sign | 0x7C00;
    int E;
    frexp(a, &E);                      /* a in [2^(E-1), 2^E) */
    int e = E - 1;
    int ulp_exp = (e < -14) ? -24 : e - 10;        /* spacing of binary16 values near a */
    double q = ldexp(a, -ulp_exp);                 /* exact: scaling by a power of two */
    double r = nearbyint(q);                       /* ties to even in the default mode */
    double v = ldexp(r, ulp_exp);
    if (v > 65504.0) return sign | 0x7C00;
    if (v < ldexp(1.0, -14))                       /* subnormal (or the first normal) */
        return sign | (uint16_t)(v / ldexp(1.0, -24));
    int E2;
    frexp(v, &E2);
    int e2 = E2 - 1;
    uint16_t frac = (uint16_t)(ldexp(v, 10 - e2) - 1024.0);
    return sign | (uint16_t)((e2 + 15) << 10) | frac;
}

/* "tensor-formats.md" section 3.1: BF16 is the high half of a binary32 word. */
double pnq_ref_bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* "tensor-formats.md" section 3.3: E2M1 has sign bit 3, exponent bits 2:1, mantissa bit 0.
 * The page prints the positive grid 0, 0.5, 1, 1.5, 2, 3, 4, 6; written here as the
 * usual minifloat rule with exponent bias 1 (e = 0 is subnormal: m * 0.5). */
double pnq_ref_e2m1_to_double(uint8_t c) {
    int sign = (c >> 3) & 1;
    int e = (c >> 1) & 3;
    int m = c & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -v : v;
}

/* "tensor-formats.md" section 3.3: E4M3FN, sign bit 7, exponent bits 6:3, fraction 2:0, bias 7. */
double pnq_ref_e4m3fn_to_double(uint8_t c) {
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 15;
    int m = c & 7;
    double v;
    if (e == 0)
        v = ldexp((double)m, -9);                  /* signed zero or m * 2^-9 */
    else if (e == 15 && m == 7)
        v = NAN;
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* ---- PN block access ("PN weight format", section Block layout) ------------ */

/* Little-endian 16-bit read at any byte offset: no alignment is assumed. */
static uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

static uint32_t rd32(const uint8_t* p) {
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

static void wr16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); }

static void wr32(uint8_t* p, uint32_t v) {
    p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); p[2] = (uint8_t)(v >> 16); p[3] = (uint8_t)(v >> 24);
}

/* Code n of element e: word e / cpw, t = e mod cpw, shift = BITS*(t>>1) + 16*(t&1). */
static int pn_code(const pn_params* p, const uint8_t* block, int e) {
    int word = e / p->cpw;
    int t = e % p->cpw;
    uint32_t w = rd32(block + 2 + 4 * word);
    int shift = p->bits * (t >> 1) + 16 * (t & 1);
    return (int)((w >> shift) & ((1u << p->bits) - 1u));
}

static int check_pn_shape(const pn_params* p, int64_t n_rows, int64_t K) {
    if (n_rows < 0 || K <= 0 || K % p->blk != 0) return 0;
    return 1;
}

/* "PN weight format", section Value: w = d * (n - z). The page states the product is exact
 * in fp32; it is formed here in fp64 and stored as fp32 (the same value when exact). The
 * sign of a zero follows the IEEE product, so code z with negative d gives -0.0. */
int pnq_ref_dequantize_row(int type, const uint8_t* W, int64_t n_rows, int64_t K, float* out) {
    pn_params p;
    if (!pn_lookup(type, &p)) return PNQ_REF_ERR_TYPE;
    if (!check_pn_shape(&p, n_rows, K)) return PNQ_REF_ERR_SHAPE;
    if ((!W || !out) && n_rows > 0) return PNQ_REF_ERR_NULL;
    int64_t nb = K / p.blk;
    for (int64_t r = 0; r < n_rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t* block = W + (r * nb + b) * 34;
            double d = pnq_ref_fp16_to_double(rd16(block));
            for (int e = 0; e < p.blk; ++e) {
                int n = pn_code(&p, block, e);
                out[r * K + b * p.blk + e] = (float)(d * (double)(n - p.z));
            }
        }
    }
    return PNQ_REF_OK;
}

/* "PN weight format", section "Where PN runs": the CPU dot product shifts by element index
 * instead of pair index and decodes most weights wrong. Kept only as a negative control. */
int pnq_ref_dequantize_row_elemshift(int type, const uint8_t* W, int64_t n_rows, int64_t K, float* out) {
    pn_params p;
    if (!pn_lookup(type, &p)) return PNQ_REF_ERR_TYPE;
    if (!check_pn_shape(&p, n_rows, K)) return PNQ_REF_ERR_SHAPE;
    if ((!W || !out) && n_rows > 0) return PNQ_REF_ERR_NULL;
    int64_t nb = K / p.blk;
    for (int64_t r = 0; r < n_rows; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t* block = W + (r * nb + b) * 34;
            double d = pnq_ref_fp16_to_double(rd16(block));
            for (int e = 0; e < p.blk; ++e) {
                uint32_t w = rd32(block + 2 + 4 * (e / p.cpw));
                int t = e % p.cpw;
                int n = (int)((w >> (p.bits * t)) & ((1u << p.bits) - 1u));
                out[r * K + b * p.blk + e] = (float)(d * (double)(n - p.z));
            }
        }
    return PNQ_REF_OK;
}

/* "PN weight format", section Validation: a row is invalid when any block's d is an fp16
 * NaN or infinity, or (pn3t) bit 15 or bit 31 of any word is set. */
int pnq_ref_validate_row(int type, const uint8_t* W, int64_t n_rows, int64_t K, int32_t* flags) {
    pn_params p;
    if (!pn_lookup(type, &p)) return PNQ_REF_ERR_TYPE;
    if (!check_pn_shape(&p, n_rows, K)) return PNQ_REF_ERR_SHAPE;
    if ((!W || !flags) && n_rows > 0) return PNQ_REF_ERR_NULL;
    int64_t nb = K / p.blk;
    for (int64_t r = 0; r < n_rows; ++r) {
        int bad = 0;
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t* block = W + (r * nb + b) * 34;
            double d = pnq_ref_fp16_to_double(rd16(block));
            if (!isfinite(d)) bad = 1;
            if (type == PNQ_REF_PN3T)
                for (int i = 0; i < 8; ++i) {
                    uint32_t w = rd32(block + 2 + 4 * i);
                    if ((w >> 15) & 1) bad = 1;
                    if ((w >> 31) & 1) bad = 1;
                }
        }
        flags[r] = bad;
    }
    return PNQ_REF_OK;
}

/* "PN weight format", section Reference quantizer, one group of BLK weights:
 *  1. amax, max, min in double; amax == 0 is the canonical zero group (d = +0, codes z).
 *  2. sigma = +1 if |min| > max else -1.
 *  3. for m in 0.50, 0.52, ..., 1.20: s = fp16(sigma * m * amax / z), skip s == 0;
 *     n = clamp(rint(w / s) + z, 0, 2z - 1); error = sum (w - s (n - z))^2 in double.
 *  4. keep the smallest error, a tie going to the larger m; d = s; reserved bits 0.
 * Readings where the page is silent: m = (50 + 2i) / 100 in double; the fp16 rounding is
 * one step from double; an s that overflows fp16 is skipped like s == 0; if every
 * candidate is skipped the group is written as the canonical zero group; non-finite
 * input is an error. */
static int quantize_block(const pn_params* p, const float* w, uint8_t* block, double* chosen_m) {
    double amax = 0.0, mx = -INFINITY, mn = INFINITY;
    for (int k = 0; k < p->blk; ++k) {
        double v = (double)w[k];
        if (!isfinite(v)) return PNQ_REF_ERR_VALUE;
        if (fabs(v) > amax) amax = fabs(v);
        if (v > mx) mx = v;
        if (v < mn) mn = v;
    }
    int codes[80];
    uint16_t dbits = 0x0000;
    double m_kept = 0.0;
    for (int k = 0; k < p->blk; ++k) codes[k] = p->z;
    if (amax != 0.0) {
        double sigma = (fabs(mn) > mx) ? 1.0 : -1.0;
        double best = INFINITY;
        int found = 0;
        for (int i = 0; i < 36; ++i) {
            double m = (50.0 + 2.0 * i) / 100.0;
            uint16_t sb = pnq_ref_double_to_fp16(sigma * m * amax / (double)p->z);
            double s = pnq_ref_fp16_to_double(sb);
            if (s == 0.0 || !isfinite(s)) continue;
            int cand[80];
            double err = 0.0;
            for (int k = 0; k < p->blk; ++k) {
                double q = nearbyint((double)w[k] / s) + (double)p->z;
                if (q < 0.0) q = 0.0;
                if (q > (double)(2 * p->z - 1)) q = (double)(2 * p->z - 1);
                cand[k] = (int)q;
                double diff = (double)w[k] - s * (double)(cand[k] - p->z);
                err += diff * diff;
            }
            if (!found || err <= best) {
                found = 1;
                best = err;
                dbits = sb;
                m_kept = m;
                for (int k = 0; k < p->blk; ++k) codes[k] = cand[k];
            }
        }
        if (!found) {
            dbits = 0x0000;
            m_kept = 0.0;
            for (int k = 0; k < p->blk; ++k) codes[k] = p->z;
        }
    }
    /* pack: element e into word e / cpw at shift BITS*(t>>1) + 16*(t&1) */
    uint32_t words[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int e = 0; e < p->blk; ++e) {
        int t = e % p->cpw;
        int shift = p->bits * (t >> 1) + 16 * (t & 1);
        words[e / p->cpw] |= (uint32_t)codes[e] << shift;
    }
    wr16(block, dbits);
    for (int i = 0; i < 8; ++i) wr32(block + 2 + 4 * i, words[i]);
    if (chosen_m) *chosen_m = m_kept;
    return PNQ_REF_OK;
}

int pnq_ref_quantize_row(int type, const float* w, int64_t K, uint8_t* out, double* chosen_m) {
    pn_params p;
    if (!pn_lookup(type, &p)) return PNQ_REF_ERR_TYPE;
    if (!check_pn_shape(&p, 1, K)) return PNQ_REF_ERR_SHAPE;
    if (!w || !out) return PNQ_REF_ERR_NULL;
    int64_t nb = K / p.blk;
    for (int64_t b = 0; b < nb; ++b) {
        int rc = quantize_block(&p, w + b * p.blk, out + b * 34, chosen_m ? chosen_m + b : NULL);
        if (rc != PNQ_REF_OK) return rc;
    }
    return PNQ_REF_OK;
}

/* ---- NVFP4 ----------------------------------------------------------------- */

/* "Quantisation and profiles", NVFP4: w = e2m1(code) * weight_scale[n, k // 16] * weight_scale_2.
 * Code k of a row sits in byte k / 2, low nibble for even k (a reading: the page is silent).
 * The represented weight is formed exactly in fp64: e2m1 * e4m3 has at most 6 significant
 * bits and the product with the fp32 global has at most 30. */
static double nvfp4_weight(const uint8_t* codes_row, const uint8_t* scales_row, float g, int64_t k) {
    uint8_t byte = codes_row[k / 2];
    uint8_t c = (k & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
    double s = pnq_ref_e4m3fn_to_double(scales_row[k / 16]);
    return pnq_ref_e2m1_to_double(c) * s * (double)g;
}

/* Dequantized fp32 value: the exact weight rounded once (to nearest even) to fp32. */
int pnq_ref_dequantize_row_nvfp4(const uint8_t* codes, const uint8_t* scales, float g,
                                 int64_t n_rows, int64_t K, float* out) {
    if (n_rows < 0 || K <= 0 || K % 16 != 0) return PNQ_REF_ERR_SHAPE;
    if ((!codes || !scales || !out) && n_rows > 0) return PNQ_REF_ERR_NULL;
    for (int64_t r = 0; r < n_rows; ++r)
        for (int64_t k = 0; k < K; ++k)
            out[r * K + k] = (float)nvfp4_weight(codes + r * (K / 2), scales + r * (K / 16), g, k);
    return PNQ_REF_OK;
}

/* "tensor-formats.md" section 3.3: stored scales admit only sign-zero finite words
 * (negative values, -0 and both NaN words are invalid); the global field must be finite
 * and strictly positive. Every E2M1 code word is valid. */
int pnq_ref_validate_row_nvfp4(const uint8_t* scales, float g, int64_t n_rows, int64_t K,
                               int32_t* flags) {
    if (n_rows < 0 || K <= 0 || K % 16 != 0) return PNQ_REF_ERR_SHAPE;
    if ((!scales || !flags) && n_rows > 0) return PNQ_REF_ERR_NULL;
    int g_ok = isfinite(g) && g > 0.0f;
    for (int64_t r = 0; r < n_rows; ++r) {
        int bad = !g_ok;
        for (int64_t j = 0; j < K / 16; ++j) {
            uint8_t s = scales[r * (K / 16) + j];
            if (s & 0x80) bad = 1;                              /* sign set: negative or -0 */
            if (isnan(pnq_ref_e4m3fn_to_double(s))) bad = 1;
        }
        flags[r] = bad;
    }
    return PNQ_REF_OK;
}

/* ---- GEMV -------------------------------------------------------------------
 * Y[m][n] = sum_k w[n][k] x[m][k] (ggml row convention), w the exact decoded weight,
 * summed in fp64 in k order; A[m][n] = sum_k |w[n][k] x[m][k]| for the tolerance
 * |y - Y| <= 1e-5 * A + 1e-6. The operator oracle starts from the exact-decoded weight
 * ("tensor-formats.md", conformance: an Op oracle starts from the represented activation
 * and the exact-decoded persistent weight). */

static void dot_rows(const float* wrow, int64_t K, const double* xd, int M, int64_t N, int64_t n,
                     double* Y, double* A) {
    for (int m = 0; m < M; ++m) {
        double s = 0.0, a = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double t = (double)wrow[k] * xd[(int64_t)m * K + k];
            s += t;
            a += fabs(t);
        }
        Y[(int64_t)m * N + n] = s;
        if (A) A[(int64_t)m * N + n] = a;
    }
}

int pnq_ref_gemv(int type, const uint8_t* W, int64_t N, int64_t K, const float* X, int M,
                 double* Y, double* A) {
    pn_params p;
    if (!pn_lookup(type, &p)) return PNQ_REF_ERR_TYPE;
    if (!check_pn_shape(&p, N, K) || M < 1) return PNQ_REF_ERR_SHAPE;
    if (!W || !X || !Y) return PNQ_REF_ERR_NULL;
    float* wrow = (float*)malloc((size_t)K * sizeof(float));
    double* xd = (double*)malloc((size_t)K * (size_t)M * sizeof(double));
    if (!wrow || !xd) { free(wrow); free(xd); return PNQ_REF_ERR_VALUE; }
    for (int64_t i = 0; i < (int64_t)M * K; ++i) xd[i] = (double)X[i];
    int64_t rowbytes = (K / p.blk) * 34;
    for (int64_t n = 0; n < N; ++n) {
        pnq_ref_dequantize_row(type, W + n * rowbytes, 1, K, wrow);
        dot_rows(wrow, K, xd, M, N, n, Y, A);
    }
    free(wrow);
    free(xd);
    return PNQ_REF_OK;
}

/* GEMV over the divisor reading: the weight is e2m1 * e4m3 (exact) divided by d_w in fp64, which
 * is within 2^-53 of the exact quotient (far inside the GEMV tolerance). */
int pnq_ref_gemv_nvfp4_div(const uint8_t* codes, const uint8_t* scales, float dw, int64_t N,
                           int64_t K, const uint16_t* X, int M, double* Y, double* A) {
    if (N < 0 || K <= 0 || K % 16 != 0 || M < 1) return PNQ_REF_ERR_SHAPE;
    if (!codes || !scales || !X || !Y) return PNQ_REF_ERR_NULL;
    double* xd = (double*)malloc((size_t)K * (size_t)M * sizeof(double));
    if (!xd) return PNQ_REF_ERR_VALUE;
    for (int64_t i = 0; i < (int64_t)M * K; ++i) xd[i] = pnq_ref_bf16_to_double(X[i]);
    for (int64_t n = 0; n < N; ++n)
        for (int m = 0; m < M; ++m) {
            double s = 0.0, a = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double w = nvfp4_weight(codes + n * (K / 2), scales + n * (K / 16), 1.0f, k) / (double)dw;
                double t = w * xd[(int64_t)m * K + k];
                s += t;
                a += fabs(t);
            }
            Y[(int64_t)m * N + n] = s;
            if (A) A[(int64_t)m * N + n] = a;
        }
    free(xd);
    return PNQ_REF_OK;
}

/* "tensor-formats.md" section 3.3 reads the global field as a divisor d_w:
 * W = e2m1(code) * e4m3fn(scale) / d_w. e2m1 * e4m3 is exact in fp32 (at most 7 significant bits,
 * magnitudes 2^-10 .. 2688), so the fp32 quotient is the exact weight rounded once. */
int pnq_ref_dequantize_row_nvfp4_div(const uint8_t* codes, const uint8_t* scales, float dw,
                                     int64_t n_rows, int64_t K, float* out) {
    if (n_rows < 0 || K <= 0 || K % 16 != 0) return PNQ_REF_ERR_SHAPE;
    if ((!codes || !scales || !out) && n_rows > 0) return PNQ_REF_ERR_NULL;
    for (int64_t r = 0; r < n_rows; ++r)
        for (int64_t k = 0; k < K; ++k) {
            float prod = (float)nvfp4_weight(codes + r * (K / 2), scales + r * (K / 16), 1.0f, k);
            out[r * K + k] = prod / dw;
        }
    return PNQ_REF_OK;
}

int pnq_ref_gemv_nvfp4(const uint8_t* codes, const uint8_t* scales, float g, int64_t N,
                       int64_t K, const uint16_t* X, int M, double* Y, double* A) {
    if (N < 0 || K <= 0 || K % 16 != 0 || M < 1) return PNQ_REF_ERR_SHAPE;
    if (!codes || !scales || !X || !Y) return PNQ_REF_ERR_NULL;
    double* xd = (double*)malloc((size_t)K * (size_t)M * sizeof(double));
    if (!xd) return PNQ_REF_ERR_VALUE;
    for (int64_t i = 0; i < (int64_t)M * K; ++i) xd[i] = pnq_ref_bf16_to_double(X[i]);
    for (int64_t n = 0; n < N; ++n)
        for (int m = 0; m < M; ++m) {
            double s = 0.0, a = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double t = nvfp4_weight(codes + n * (K / 2), scales + n * (K / 16), g, k) *
                           xd[(int64_t)m * K + k];
                s += t;
                a += fabs(t);
            }
            Y[(int64_t)m * N + n] = s;
            if (A) A[(int64_t)m * N + n] = a;
        }
    free(xd);
    return PNQ_REF_OK;
}

/* ---- grouped signed-integer formats ("tensor-formats.md", sections 4 to 7) ----------------
 * Q4G64_F16S, Q5G64_F16S, Q6G64_F16S (b = 4, 5, 6 bits, groups of G = 64) and W8G32_F16S
 * (b = 8, G = 32): one two's-complement code per weight, one binary16 scale per group of G along
 * K (the last group of a row may be partial), reconstruction w = binary32(s32 * binary32(q)).
 *
 * Physical layout (the pages leave it to a layout registry; this is the library's own, a
 * reading): K % 8 == 0; the low 4 bits of each logical word u in a nibble plane lo[N][K/2]
 * (even k in the low nibble); the bits above in a second plane hi: Q5 one bit per weight,
 * hi[N][K/8], bit k % 8 of byte k / 8; Q6 two bits per weight, hi[N][K/4], bits
 * 2 (k % 4) .. 2 (k % 4) + 1 of byte k / 4; W8 stores u as one byte per weight in lo[N][K]
 * and has no hi plane. Scales sc[N][ceil(K / G)], binary16 words. */

typedef struct {
    int bits, G, qmin, qmax;
} grp_params;

static int grp_lookup(int type, grp_params* p) {
    switch (type) {
        case PNQ_REF_Q4G64: p->bits = 4; p->G = 64; p->qmin = -8; p->qmax = 7; return 1;
        case PNQ_REF_Q5G64: p->bits = 5; p->G = 64; p->qmin = -16; p->qmax = 15; return 1;
        case PNQ_REF_Q6G64: p->bits = 6; p->G = 64; p->qmin = -32; p->qmax = 31; return 1;
        case PNQ_REF_W8G32: p->bits = 8; p->G = 32; p->qmin = -127; p->qmax = 127; return 1;
        default: return 0;
    }
}

/* Logical word u of weight k of a row (planes of that row). */
static uint32_t grp_word(const grp_params* p, const uint8_t* lo, const uint8_t* hi, int64_t k) {
    if (p->bits == 8) return lo[k];
    uint32_t u = (k & 1) ? (uint32_t)(lo[k / 2] >> 4) : (uint32_t)(lo[k / 2] & 15);
    if (p->bits == 5) u |= (uint32_t)((hi[k / 8] >> (k % 8)) & 1) << 4;
    if (p->bits == 6) u |= (uint32_t)((hi[k / 4] >> (2 * (k % 4))) & 3) << 4;
    return u;
}

static void grp_put(const grp_params* p, uint8_t* lo, uint8_t* hi, int64_t k, uint32_t u) {
    if (p->bits == 8) { lo[k] = (uint8_t)u; return; }
    if (k & 1) lo[k / 2] = (uint8_t)((lo[k / 2] & 0x0F) | ((u & 15) << 4));
    else lo[k / 2] = (uint8_t)((lo[k / 2] & 0xF0) | (u & 15));
    if (p->bits == 5) hi[k / 8] = (uint8_t)((hi[k / 8] & ~(1u << (k % 8))) | (((u >> 4) & 1) << (k % 8)));
    if (p->bits == 6)
        hi[k / 4] = (uint8_t)((hi[k / 4] & ~(3u << (2 * (k % 4)))) | (((u >> 4) & 3) << (2 * (k % 4))));
}

/* Section 5: q = u for u < 2^(b-1), else u - 2^b. */
static int grp_signed(const grp_params* p, uint32_t u) {
    return (u < (1u << (p->bits - 1))) ? (int)u : (int)u - (1 << p->bits);
}

int pnq_ref_grouped_plane_bytes(int type, int64_t K, int64_t* lo_bytes, int64_t* hi_bytes, int64_t* n_scales) {
    grp_params p;
    if (!grp_lookup(type, &p)) return PNQ_REF_ERR_TYPE;
    if (K <= 0 || K % 8 != 0) return PNQ_REF_ERR_SHAPE;
    *lo_bytes = (p.bits == 8) ? K : K / 2;
    *hi_bytes = (p.bits == 5) ? K / 8 : (p.bits == 6) ? K / 4 : 0;
    *n_scales = (K + p.G - 1) / p.G;
    return PNQ_REF_OK;
}

static float f16_bits_to_float(uint16_t h) { return (float)pnq_ref_fp16_to_double(h); } /* exact */

/* Section 6.2: w_hat = binary32(s32 * binary32(q)). */
int pnq_ref_dequantize_grouped(int type, const uint8_t* lo, const uint8_t* hi, const uint16_t* sc,
                               int64_t n_rows, int64_t K, float* out) {
    grp_params p;
    int64_t lb, hb, ns;
    int rc = pnq_ref_grouped_plane_bytes(type, K, &lb, &hb, &ns);
    if (rc != PNQ_REF_OK) return rc;
    grp_lookup(type, &p);
    if (n_rows < 0) return PNQ_REF_ERR_SHAPE;
    if (n_rows > 0 && (!lo || !sc || !out || (hb > 0 && !hi))) return PNQ_REF_ERR_NULL;
    for (int64_t r = 0; r < n_rows; ++r)
        for (int64_t k = 0; k < K; ++k) {
            int q = grp_signed(&p, grp_word(&p, lo + r * lb, hi ? hi + r * hb : NULL, k));
            float s32 = f16_bits_to_float(sc[r * ns + k / p.G]);
            out[r * K + k] = s32 * (float)q;
        }
    return PNQ_REF_OK;
}

/* Section 6 validity: a scale is +0 or a finite positive binary16 (sign clear, exponent not all
 * ones); a group whose scale is +0 holds only zero codes; W8 never holds the word 0x80. */
int pnq_ref_validate_grouped(int type, const uint8_t* lo, const uint8_t* hi, const uint16_t* sc,
                             int64_t n_rows, int64_t K, int32_t* flags) {
    grp_params p;
    int64_t lb, hb, ns;
    int rc = pnq_ref_grouped_plane_bytes(type, K, &lb, &hb, &ns);
    if (rc != PNQ_REF_OK) return rc;
    grp_lookup(type, &p);
    if (n_rows < 0) return PNQ_REF_ERR_SHAPE;
    if (n_rows > 0 && (!lo || !sc || !flags || (hb > 0 && !hi))) return PNQ_REF_ERR_NULL;
    for (int64_t r = 0; r < n_rows; ++r) {
        int bad = 0;
        for (int64_t k = 0; k < K; ++k) {
            uint16_t s = sc[r * ns + k / p.G];
            uint32_t u = grp_word(&p, lo + r * lb, hi ? hi + r * hb : NULL, k);
            if ((s & 0x8000) || (s & 0x7C00) == 0x7C00) bad = 1;
            if (s == 0 && u != 0) bad = 1;
            if (p.bits == 8 && u == 0x80) bad = 1;
        }
        flags[r] = bad;
    }
    return PNQ_REF_OK;
}

/* Section 7, MAXABS_F16_RECIP_RNE_V1, per group of binary32 values, every step rounded to
 * nearest even in binary32 (or binary16 for the scale):
 *   amax = max |x|; amax == +0 -> scale +0, codes 0;
 *   raw = amax / qmax; scale16 = binary16(raw), +0 -> 0x0001; not finite -> fail;
 *   inv = 1 / scale32; code = clamp(rint(x * inv), qmin, qmax).
 * A non-finite source value fails. On failure the call returns PNQ_REF_ERR_VALUE and
 * fail_row (if given) receives the row. */
int pnq_ref_quantize_grouped(int type, const float* w, int64_t n_rows, int64_t K, uint8_t* lo,
                             uint8_t* hi, uint16_t* sc, int64_t* fail_row) {
    grp_params p;
    int64_t lb, hb, ns;
    int rc = pnq_ref_grouped_plane_bytes(type, K, &lb, &hb, &ns);
    if (rc != PNQ_REF_OK) return rc;
    grp_lookup(type, &p);
    if (n_rows < 0) return PNQ_REF_ERR_SHAPE;
    if (n_rows > 0 && (!w || !lo || !sc || (hb > 0 && !hi))) return PNQ_REF_ERR_NULL;
    for (int64_t r = 0; r < n_rows; ++r) {
        uint8_t* lr = lo + r * lb;
        uint8_t* hr = hi ? hi + r * hb : NULL;
        for (int64_t g = 0; g < ns; ++g) {
            int64_t k0 = g * p.G, k1 = (k0 + p.G < K) ? k0 + p.G : K;
            float amax = 0.0f;
            for (int64_t k = k0; k < k1; ++k) {
                float v = w[r * K + k];
                if (!isfinite(v)) { if (fail_row) *fail_row = r; return PNQ_REF_ERR_VALUE; }
                if (fabsf(v) > amax) amax = fabsf(v);
            }
            if (amax == 0.0f) {
                sc[r * ns + g] = 0x0000;
                for (int64_t k = k0; k < k1; ++k) grp_put(&p, lr, hr, k, 0);
                continue;
            }
            float raw = amax / (float)p.qmax;
            uint16_t s16 = pnq_ref_double_to_fp16((double)raw);  /* one rounding: raw is exact in fp64 */
            if (s16 == 0x0000) s16 = 0x0001;
            if ((s16 & 0x7C00) == 0x7C00) { if (fail_row) *fail_row = r; return PNQ_REF_ERR_VALUE; }
            sc[r * ns + g] = s16;
            float inv = 1.0f / f16_bits_to_float(s16);
            for (int64_t k = k0; k < k1; ++k) {
                float nrm = w[r * K + k] * inv;
                float q = rintf(nrm);  /* ties to even in the default rounding mode */
                if (q < (float)p.qmin) q = (float)p.qmin;
                if (q > (float)p.qmax) q = (float)p.qmax;
                int qi = (int)q;
                grp_put(&p, lr, hr, k, (uint32_t)qi & ((1u << p.bits) - 1u));
            }
        }
    }
    return PNQ_REF_OK;
}

/* Y[m][n] = sum_k w_hat[n][k] x[m][k] in fp64 over the reconstructed binary32 weights, x fp32. */
int pnq_ref_gemv_grouped(int type, const uint8_t* lo, const uint8_t* hi, const uint16_t* sc, int64_t N,
                         int64_t K, const float* X, int M, double* Y, double* A) {
    int64_t lb, hb, ns;
    int rc = pnq_ref_grouped_plane_bytes(type, K, &lb, &hb, &ns);
    if (rc != PNQ_REF_OK) return rc;
    if (N < 0 || M < 1) return PNQ_REF_ERR_SHAPE;
    if (!lo || !sc || !X || !Y || (hb > 0 && !hi)) return PNQ_REF_ERR_NULL;
    float* row = (float*)malloc((size_t)K * sizeof(float));
    double* xd = (double*)malloc((size_t)K * (size_t)M * sizeof(double));
    if (!row || !xd) { free(row); free(xd); return PNQ_REF_ERR_VALUE; }
    for (int64_t i = 0; i < (int64_t)M * K; ++i) xd[i] = (double)X[i];
    for (int64_t n = 0; n < N; ++n) {
        pnq_ref_dequantize_grouped(type, lo + n * lb, hi ? hi + n * hb : NULL, sc + n * ns, 1, K, row);
        dot_rows(row, K, xd, M, N, n, Y, A);
    }
    free(row);
    free(xd);
    return PNQ_REF_OK;
}

/* ---- NVFP4 clip search (TandemLLM "Quantisation and profiles", section "The clip search") ------
 * Per group of 16 weights of a row, five scale multipliers 1.00, 0.95, 0.90, 0.85, 0.80 are
 * tried and the one with the smallest error  sum_k act_ms[k] (w[k] - dequant(quant(w[k])))^2
 * is kept. Readings where the page is silent (the page's tool is not printed): the weight is
 * e2m1 * e4m3 * g with a given global multiplier g (the TandemLLM reading); the multiplier
 * scales the group's base scale amax / (6 g) (6: the largest e2m1 magnitude), computed in
 * double as ((mu * amax) / 6) / g; the scale is the nearest E4M3FN value, ties to the even code
 * word, saturating at 448; each weight takes the nearest E2M1 magnitude of |w| / (scale * g),
 * ties to the even code word, saturating at 6, with the sign of w (a negative weight that rounds
 * to zero keeps the negative-zero word); a zero scale gives every weight the zero word of its
 * sign; the error is summed in k order in double; a tie in error keeps the earlier multiplier.
 * Every step is one IEEE double operation in that order. */

static const double kClipMultipliers[5] = {1.00, 0.95, 0.90, 0.85, 0.80};

/* Nearest positive E4M3FN code word to t >= 0 (0x00 .. 0x7E), ties to the even word. */
static uint8_t e4m3_nearest(double t) {
    uint8_t best = 0;
    double bd = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double d = fabs(pnq_ref_e4m3fn_to_double((uint8_t)c) - t);
        if (d < bd || (d == bd && (c & 1) == 0)) { bd = d; best = (uint8_t)c; }
    }
    return best;
}

/* Nearest E2M1 magnitude word (0..7) to a >= 0, ties to the even word. */
static uint8_t e2m1_nearest(double a) {
    uint8_t best = 0;
    double bd = INFINITY;
    for (int c = 0; c <= 7; ++c) {
        double d = fabs(pnq_ref_e2m1_to_double((uint8_t)c) - a);
        if (d < bd || (d == bd && (c & 1) == 0)) { bd = d; best = (uint8_t)c; }
    }
    return best;
}

int pnq_ref_quantize_nvfp4_clip(const float* w, const float* act_ms, float g, int64_t n_rows, int64_t K,
                                uint8_t* codes, uint8_t* scales, int32_t* chosen) {
    if (n_rows < 0 || K <= 0 || K % 16 != 0) return PNQ_REF_ERR_SHAPE;
    if (n_rows > 0 && (!w || !act_ms || !codes || !scales)) return PNQ_REF_ERR_NULL;
    if (!(isfinite(g) && g > 0.0f)) return PNQ_REF_ERR_VALUE;
    const double gd = (double)g;
    for (int64_t r = 0; r < n_rows; ++r)
        for (int64_t grp = 0; grp < K / 16; ++grp) {
            const float* x = w + r * K + grp * 16;
            const float* a = act_ms + grp * 16;
            double amax = 0.0;
            for (int k = 0; k < 16; ++k) {
                if (!isfinite(x[k])) return PNQ_REF_ERR_VALUE;
                if (fabs((double)x[k]) > amax) amax = fabs((double)x[k]);
            }
            double best = INFINITY;
            int best_i = 0;
            uint8_t best_sc = 0, best_c[16];
            for (int i = 0; i < 5; ++i) {
                double t = ((kClipMultipliers[i] * amax) / 6.0) / gd;
                uint8_t sc = e4m3_nearest(t);
                double sv = pnq_ref_e4m3fn_to_double(sc);
                uint8_t cw[16];
                double err = 0.0;
                for (int k = 0; k < 16; ++k) {
                    uint8_t sign = (x[k] < 0.0f || (x[k] == 0.0f && signbit(x[k]))) ? 8 : 0;
                    uint8_t mag = 0;
                    if (sv != 0.0) mag = e2m1_nearest(fabs((double)x[k]) / (sv * gd));
                    cw[k] = (uint8_t)(sign | mag);
                    double dq = (pnq_ref_e2m1_to_double(cw[k]) * sv) * gd;
                    double diff = (double)x[k] - dq;
                    err = err + (double)a[k] * (diff * diff);
                }
                if (i == 0 || err < best) {
                    best = err;
                    best_i = i;
                    best_sc = sc;
                    memcpy(best_c, cw, sizeof cw);
                }
            }
            scales[r * (K / 16) + grp] = best_sc;
            for (int k = 0; k < 16; k += 2)
                codes[r * (K / 2) + grp * 8 + k / 2] = (uint8_t)(best_c[k] | (best_c[k + 1] << 4));
            if (chosen) chosen[r * (K / 16) + grp] = best_i;
        }
    return PNQ_REF_OK;
}
