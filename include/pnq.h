/*
 * pnq.h -- C ABI of libpnq: decode-time products straight from block-quantized
 * weights (pn3t, pn4t, NVFP4 W4A16) on sm_103a (GB300).
 *
 * Conventions shared by every entry point
 *   - Returns PNQ_OK (0) or a negative pnq_status. Nothing aborts; no kernel traps.
 *   - Device pointers are plain CUDA device addresses owned by the caller. The library
 *     allocates no device memory in any entry point: the fast GEMV paths sum their partial
 *     results on chip (shared memory, and distributed shared memory between the two CTAs of
 *     a thread-block cluster), so calls may be made from any stream, during stream capture,
 *     and from several host threads at once.
 *   - Calls are asynchronous and ordered on `stream` (0 = the legacy default stream).
 *     Argument errors are reported before anything is launched; a launch failure is
 *     reported as PNQ_ERR_CUDA. Results are valid once the stream reaches the call.
 *   - Matrices are row-major with the ggml row convention: weight row n holds the K
 *     weights that multiply x[m][0..K), so Y[m][n] = sum_k W[n][k] * X[m][k].
 *   - Y / out / flags are overwritten, never accumulated into.
 *
 * Weight formats (citations name the page and its section)
 *   PNQ_PN3T (124), PNQ_PN4T (125): "PN weight format" (tensorless docs, reference/pn-format),
 *     sections Types, Block layout and Value. A row of K weights is K/BLK consecutive
 *     34-byte blocks (BLK = 80 for pn3t, 64 for pn4t); rows are back to back, so row n
 *     starts at byte n * (K/BLK) * 34. A block is d (fp16, little-endian, signed) at bytes
 *     0..1 and eight little-endian u32 words at bytes 2..33; element e is in word
 *     e / CPW (CPW = 10 or 8) at shift BITS*(t>>1) + 16*(t&1), t = e mod CPW, and
 *     decodes to w = d * (n - z), z = 4 (pn3t) or 8 (pn4t). W needs only 2-byte
 *     alignment: odd blocks' words are not 4-byte aligned.
 *   PNQ_NVFP4 (1004, a library id; the pages assign none): TandemLLM "Quantisation and
 *     profiles", section NVFP4, and NInfer "tensor-formats.md" section 3.3. Weight
 *     w[n][k] = e2m1(code[n][k]) * e4m3fn(scale[n][k/16]) * global_scale, with codes
 *     packed two per byte, low nibble = even k, [N][K/2] row-major, and scales one
 *     E4M3FN byte per 16 weights along K, [N][K/16] row-major. global_scale is a
 *     multiplier (the TandemLLM reading).
 *   PNQ_NVFP4_DIV (1005, a library id): the same codes and scales with the global field read
 *     as a divisor d_w ("tensor-formats.md" section 3.3): w = e2m1 * e4m3fn / d_w. The
 *     pnq_nvfp4_weights descriptor carries d_w in global_scale.
 *   PNQ_Q4G64_F16S, PNQ_Q5G64_F16S, PNQ_Q6G64_F16S, PNQ_W8G32_F16S (1104, 1105, 1106, 1108,
 *     library ids): the grouped signed-integer formats of NInfer "tensor-formats.md" (sections 4
 *     to 7). One two's-complement code per weight (4, 5, 6 or 8 bits; W8 in -127..127) and one
 *     binary16 scale per group of 64 (32 for W8) along K, the last group of a row possibly
 *     partial; w = binary32(scale * code). K % 8 == 0. Planes (a layout of this library; the
 *     pages leave layouts to a registry), passed in a pnq_grouped_weights descriptor:
 *       lo      [N][K/2] bytes: low 4 bits of each code's word, even k in the low nibble
 *               (W8: [N][K], the code's byte);
 *       hi      Q5: [N][K/8], bit 4 of weight k at bit k % 8 of byte k / 8;
 *               Q6: [N][K/4], bits 4..5 of weight k at bits 2 (k % 4) .. of byte k / 4;
 *               Q4, W8: unused (may be NULL);
 *       scales  [N][ceil(K / G)] binary16 words.
 *     Alignment: lo 8 bytes (W8) or 4 bytes, hi 2 bytes, scales 2 bytes (else PNQ_ERR_ALIGN).
 *
 * Fast paths (taken automatically, never required)
 *   PN: W and X 16-byte aligned and (K/BLK) % 8 == 0.  NVFP4: codes, scales and X 16-byte
 *   aligned and K % 256 == 0. Other layouts run a slower (generic) path within the same
 *   accuracy bound; it is several times slower, so callers who care about speed should
 *   allocate W and X with 16-byte alignment (any cudaMalloc result is 256-byte aligned).
 */
#ifndef PNQ_H
#define PNQ_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

enum pnq_type {
    PNQ_PN3T = 124,
    PNQ_PN4T = 125,
    PNQ_NVFP4 = 1004,
    PNQ_NVFP4_DIV = 1005,
    PNQ_Q4G64_F16S = 1104,
    PNQ_Q5G64_F16S = 1105,
    PNQ_Q6G64_F16S = 1106,
    PNQ_W8G32_F16S = 1108
};

enum pnq_status {
    PNQ_OK = 0,
    PNQ_ERR_TYPE = -1,   /* unknown type id */
    PNQ_ERR_SHAPE = -2,  /* K not a positive multiple of BLK (PN) or 16 (NVFP4); N < 0;
                            M outside [1, 16]; size overflow */
    PNQ_ERR_NULL = -3,   /* a required pointer is NULL */
    PNQ_ERR_ALIGN = -4,  /* a pointer misses its minimum alignment (see each call) */
    PNQ_ERR_CUDA = -5,   /* a CUDA call failed (launch error, no device, bad stream) */
    PNQ_ERR_DEVICE = -6, /* a kernel gave up on an internal wait (see pnq_device_error) */
    PNQ_ERR_FLAGS = -7,  /* unknown bit in a flags argument */
    PNQ_ERR_SCRATCH = -8, /* the caller's scratch holds less than the call needs (pnq_gemm) */
    PNQ_ERR_VALUE = -9    /* an argument value outside its domain (a global scale that is not finite
                             and > 0) */
};

/* Flags of pnq_gemv_ex. */
enum pnq_gemv_flags {
    /* The weights are not written by any work queued earlier on the stream (e.g. model weights
     * in a decode loop). The kernel may then start streaming them from HBM while the previous
     * grid in the stream is still running; x is still read only after that grid completes. */
    PNQ_GEMV_STATIC_WEIGHTS = 1u
};

/* NVFP4 weight descriptor, passed by HOST pointer as the W argument when type ==
 * PNQ_NVFP4. codes and scales are device pointers (1-byte alignment suffices). */
typedef struct pnq_nvfp4_weights {
    const uint8_t* codes;   /* device, [N][K/2] E2M1 pairs, low nibble = even k */
    const uint8_t* scales;  /* device, [N][K/16] E4M3FN */
    float global_scale;     /* host value: multiplies every weight (PNQ_NVFP4), or the
                               divisor d_w of every weight (PNQ_NVFP4_DIV) */
} pnq_nvfp4_weights;

/* Grouped signed-integer weight descriptor, passed by HOST pointer as the W argument for the
 * PNQ_Q*G64_F16S / PNQ_W8G32_F16S types; the planes are device pointers. */
typedef struct pnq_grouped_weights {
    const uint8_t* lo;       /* device, low-4-bit plane (W8: the code bytes) */
    const uint8_t* hi;       /* device, high-bit plane (Q5, Q6), else unused */
    const uint16_t* scales;  /* device, binary16 scale per group */
} pnq_grouped_weights;

/* The same planes as outputs of pnq_quantize_row. */
typedef struct pnq_grouped_planes {
    uint8_t* lo;
    uint8_t* hi;
    uint16_t* scales;
} pnq_grouped_planes;

/*
 * pnq_gemv -- Y[m][n] = sum_k W[n][k] * X[m][k] for m < M, n < N, fp32 accumulation.
 * The decode-step product of the pages ("PN weight format", section "Where PN runs":
 * PN tensors use their own GEMV kernels; TandemLLM "Quantisation and profiles",
 * section NVFP4: the W4A16 kernel unpacks codes in registers before the multiply).
 *   type  PNQ_PN3T, PNQ_PN4T, PNQ_NVFP4, PNQ_NVFP4_DIV or a grouped signed-integer type.
 *   W     PN: device pointer to N*(K/BLK)*34 bytes, >= 2-byte aligned (else PNQ_ERR_ALIGN).
 *         NVFP4, NVFP4_DIV: host pointer to a pnq_nvfp4_weights.
 *         Grouped: host pointer to a pnq_grouped_weights (the GEMV runs on the CUDA cores; X
 *         fp32, 16-byte aligned).
 *   N     output rows (>= 0; N == 0 launches nothing).  K: inner dimension.
 *   X     device, [M][K] row-major: fp32 for PN (4-byte aligned), bf16 for NVFP4
 *         (2-byte aligned). Finite values; any magnitude is accepted.
 *   M     1..16 activation rows (1..4 per matrix-vector pass, 5..16 small batch).
 *   Y     device, [M][N] fp32, 4-byte aligned; must not overlap W or X.
 * Accuracy: |Y - Y_exact| <= 1e-5 * sum_k |W[n][k] X[m][k]| + 1e-6 for finite inputs,
 * where Y_exact is the fp64 sum over the exactly decoded weights. Weights that fail
 * pnq_validate_row give unspecified (but memory-safe) results.
 */
int pnq_gemv(int type, const void* W, int64_t N, int64_t K, const void* X, int M, float* Y,
             cudaStream_t stream);

/*
 * pnq_gemv_ex -- pnq_gemv with flags (a bitwise OR of pnq_gemv_flags; 0 = pnq_gemv).
 * Same arguments, results and errors as pnq_gemv, plus PNQ_ERR_FLAGS for unknown bits. The
 * pages define no such call: it exposes an overlap that only the caller can declare safe.
 * Launches on the fast path use programmatic dependent launch: a GEMV may begin while the
 * previous kernel on the stream finishes, and reads nothing that kernel may write (x, and
 * the weights unless PNQ_GEMV_STATIC_WEIGHTS) before that kernel has completed.
 */
int pnq_gemv_ex(int type, const void* W, int64_t N, int64_t K, const void* X, int M, float* Y,
                unsigned int flags, cudaStream_t stream);

/*
 * pnq_gemv_noalloc -- pnq_gemv_ex that allocates nothing. The pages have no counterpart; it is
 * for callers that cannot call cudaMalloc: code running under a caching or arena allocator that
 * owns all device memory, a section being captured into a graph where a first-time allocation
 * must not happen, or a runtime that forbids allocation after start-up. Same arguments, results
 * (bit for bit) and errors as pnq_gemv_ex.
 *   Scratch: none. The fast paths keep every partial sum on chip (see the conventions above),
 *   so this entry point runs exactly the kernels pnq_gemv_ex runs; it stays as the name a
 *   caller can hold the library to: whatever later versions add, it will never allocate, and it
 *   never returns PNQ_ERR_SCRATCH in this version. Calls on different streams may overlap.
 */
int pnq_gemv_noalloc(int type, const void* W, int64_t N, int64_t K, const void* X, int M, float* Y,
                     unsigned int flags, cudaStream_t stream);

/*
 * pnq_gemm -- Y[m][n] = sum_k W[n][k] * X[m][k] for any number M >= 1 of activation rows
 * (prefill), PN3T and PN4T, on the tcgen05 tensor cores. The prefill route of the pages (feedman.me
 * post on BF16_P12, section "How the engine uses it": with more than 16 tokens a cache-sized piece
 * of the weights is unpacked, then multiplied densely): the weights are decoded slice by slice into
 * the caller's scratch as two tf32 planes (the exact decoded weight is their sum) and multiplied,
 * with x split into two tf32 planes the same way, by three tf32 MMAs per K step accumulated in fp32.
 *   W        device, as for pnq_gemv (>= 2-byte aligned).
 *   X        device fp32 [M][K], 16-byte aligned.   Y: device fp32 [M][N], 4-byte aligned.
 *   scratch  device, 16-byte aligned, scratch_bytes long: 8*M*K bytes for x plus 8*K bytes per
 *            weight row of a slice; slices are the largest multiple of 128 rows that fits (at least
 *            128, else PNQ_ERR_SCRATCH). pnq_gemm_scratch_bytes gives the size for a slice length.
 *            The library allocates nothing; scratch contents are overwritten.
 * Accuracy: the pnq_gemv bound. Errors: PNQ_ERR_TYPE (NVFP4 and grouped types have no prefill
 * path here), PNQ_ERR_SHAPE, PNQ_ERR_NULL, PNQ_ERR_ALIGN, PNQ_ERR_SCRATCH, PNQ_ERR_CUDA.
 */
int pnq_gemm(int type, const void* W, int64_t N, int64_t K, const float* X, int64_t M, float* Y, void* scratch,
             uint64_t scratch_bytes, cudaStream_t stream);

/* Scratch bytes pnq_gemm needs for slices of slice_rows weight rows (rounded up to a multiple of
 * 128; 0 = all N rows in one slice). Returns PNQ_OK, PNQ_ERR_TYPE, PNQ_ERR_SHAPE or PNQ_ERR_NULL. */
int pnq_gemm_scratch_bytes(int type, int64_t N, int64_t K, int64_t M, int64_t slice_rows, uint64_t* bytes);

/*
 * pnq_dequantize_row -- out[r][k] = the fp32 weight, bit-exact:
 *   PN: fp32(d) * fp32(n - z), exact ("PN weight format", section Value: both steps exact
 *   in fp32; code z with negative d gives -0.0). NVFP4: e2m1 * e4m3 (exact) times the
 *   global scale, rounded once to nearest-even fp32. NVFP4_DIV: e2m1 * e4m3 (exact)
 *   divided by d_w, rounded once to nearest-even fp32. A non-finite d or a NaN scale gives
 *   NaN/inf of the IEEE product (bit patterns of NaNs are not specified).
 *   W      as for pnq_gemv (n_rows rows).   out: device fp32 [n_rows][K], 4-byte aligned.
 */
int pnq_dequantize_row(int type, const void* W, int64_t n_rows, int64_t K, float* out,
                       cudaStream_t stream);

/*
 * pnq_validate_row -- flags[r] = 1 if row r is invalid, else 0.
 *   Grouped ("tensor-formats.md" section 6): a scale with its sign bit set or an all-ones
 *   exponent (negative, -0, infinity, NaN), a +0 scale over a nonzero code, or (W8) the word
 *   0x80.
 *   PN ("PN weight format", section Validation): any block's d is an fp16 NaN or infinity,
 *   or (pn3t) bit 15 or bit 31 of any word is set.
 *   NVFP4 and NVFP4_DIV ("tensor-formats.md" section 3.3): any scale byte has its sign bit
 *   set (negative or -0) or is NaN (0x7F / 0xFF), or global_scale is not finite and > 0
 *   (then every row).
 *   W as for pnq_gemv.   flags: device int32 [n_rows], 4-byte aligned.
 */
int pnq_validate_row(int type, const void* W, int64_t n_rows, int64_t K, int32_t* flags,
                     cudaStream_t stream);

/*
 * pnq_quantize_row -- encode n_rows rows of K fp32 weights (device w, [n_rows][K], 4-byte
 * aligned) on the GPU; row_status (device int32 [n_rows], 4-byte aligned) is set to 0 for each
 * row encoded and 1 for a row the encoder rejects (its output bytes are then unspecified).
 *   PN3T / PN4T: the reference quantizer of "PN weight format" (section Reference quantizer),
 *     bit for bit the CPU reference's d and codes: per block, 36 multipliers 0.50 .. 1.20 of
 *     amax / z with the sign that favours the larger tail, each scale rounded to fp16, codes
 *     rint(w / s) + z clamped, the least squared error kept (a tie to the larger multiplier),
 *     all in IEEE double in that order. out: device pointer to n_rows*(K/BLK)*34 bytes, 2-byte
 *     aligned. A row with a non-finite weight is rejected.
 *   Grouped: the canonical encoder MAXABS_F16_RECIP_RNE_V1 ("tensor-formats.md" section 7):
 *     per group amax, scale16 = binary16(amax / qmax) (+0 becomes 0x0001), inv = 1 / scale,
 *     code = clamp(rint(w * inv)), each step one binary32 (binary16) rounding to nearest even;
 *     an all-zero group gets scale +0. out: host pointer to a pnq_grouped_planes. A row with a
 *     non-finite weight or a scale that overflows binary16 is rejected.
 *   Errors: PNQ_ERR_TYPE (NVFP4 types have no encoder here), PNQ_ERR_SHAPE, PNQ_ERR_NULL,
 *   PNQ_ERR_ALIGN, PNQ_ERR_CUDA. (Library call; the pages define the algorithms, not the call.)
 */
int pnq_quantize_row(int type, const float* w, int64_t n_rows, int64_t K, void* out, int32_t* row_status,
                     cudaStream_t stream);

/*
 * pnq_quantize_nvfp4_clip -- encode n_rows rows of K fp32 weights (device w, [n_rows][K]) as NVFP4
 * (codes [n_rows][K/2], scales [n_rows][K/16], device) for the global multiplier global_scale
 * with the clip search of TandemLLM "Quantisation and profiles" (section "The clip search"): per
 * group of 16, the scale multiplier among 1.00, 0.95, 0.90, 0.85, 0.80 of amax / (6 g) whose
 * act_ms-weighted squared error is smallest; act_ms (device fp32 [K]) is the mean square of each
 * input channel over calibration data. Bit for bit the CPU reference's choice. Readings where the
 * page is silent: scales round to the nearest E4M3FN value (ties to the even word, saturating at
 * 448), weights to the nearest E2M1 magnitude (ties to the even word, saturating at 6) with the
 * sign of w, the error is summed in k order in double, a tie keeps the earlier multiplier.
 * row_status (device int32 [n_rows]): 0, or 1 for a row with a non-finite weight (its bytes are
 * then unspecified). w, act_ms and row_status 4-byte aligned. Errors: PNQ_ERR_SHAPE (K % 16),
 * PNQ_ERR_VALUE (global_scale not finite and > 0), PNQ_ERR_NULL, PNQ_ERR_ALIGN, PNQ_ERR_CUDA.
 */
int pnq_quantize_nvfp4_clip(const float* w, const float* act_ms, int64_t n_rows, int64_t K, float global_scale,
                            uint8_t* codes, uint8_t* scales, int32_t* row_status, cudaStream_t stream);

/*
 * pnq_device_error -- reads and clears the library's device error word on the current
 * device (synchronous: waits for all work on the device; not for use during stream capture).
 * *code = 0 when no kernel has given up on a bounded internal wait since the last call;
 * otherwise the nonzero site code of the first one (1: a consumer's wait for a weight stage or
 * for the operands of a K unit, 2: the producer's wait for a free stage, 3: the producer's final
 * wait for copies in flight, 5: a builder's wait for a free operand slot, 6: pnq_selftest_wait),
 * and the call returns
 * PNQ_ERR_DEVICE. The Y of a GEMV that gave up is unspecified; later GEMVs are unaffected (no
 * state outlives a launch). Other returns: PNQ_OK, PNQ_ERR_NULL, PNQ_ERR_CUDA. (Library
 * plumbing; the pages define no such call.)
 */
int pnq_device_error(int32_t* code);

/*
 * pnq_selftest_wait -- exercises the failure path of the bounded waits: one thread waits, with the
 * GEMV kernels' own bounded wait limited to limit_us microseconds (1 .. 2,000,000), on a
 * shared-memory barrier that nothing arrives at, gives up and records site code 6 in the device
 * error word, as a GEMV kernel records a wait that gave up. Nothing faults or hangs: the kernel
 * returns and the context stays usable; read the code with pnq_device_error. Returns PNQ_OK,
 * PNQ_ERR_VALUE (limit out of range) or PNQ_ERR_CUDA. (Library plumbing; the pages define no such
 * call.)
 */
int pnq_selftest_wait(uint32_t limit_us, cudaStream_t stream);

/* Library version string (static storage). */
const char* pnq_version(void);

#ifdef __cplusplus
}
#endif
#endif /* PNQ_H */
