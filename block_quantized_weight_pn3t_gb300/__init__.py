"""pnq: block-quantized weight GEMV (pn3t, pn4t, NVFP4 W4A16, grouped signed-integer formats)
for sm_103a.

The compute path is the C-ABI library ``libpnq.so`` built from ``csrc/``; this
package only marshals arguments to it (see ``_binding``). Importing the package
does not load the library; the first call does, and raises if it is missing.
"""
from ._binding import (PN3T, PN4T, NVFP4, NVFP4_DIV, Q4G64_F16S, Q5G64_F16S, Q6G64_F16S, W8G32_F16S, GROUPED,
                       BLOCK_WEIGHTS, GEMV_STATIC_WEIGHTS, Status, PnqError, lib, lib_path, gemv,
                       gemv_ex_ptr, gemv_noalloc, gemv_noalloc_ptr, grouped_plane_shapes,
                       dequantize_row, validate_row, quantize_row, gemv_ptr, dequantize_row_ptr, validate_row_ptr,
                       quantize_row_ptr, quantize_nvfp4_clip, selftest_wait, gemm, gemm_scratch_bytes, device_error, nvfp4_weights, pnq_grouped_weights)

__all__ = ["PN3T", "PN4T", "NVFP4", "NVFP4_DIV", "Q4G64_F16S", "Q5G64_F16S", "Q6G64_F16S", "W8G32_F16S", "GROUPED",
           "BLOCK_WEIGHTS", "GEMV_STATIC_WEIGHTS", "gemv_ex_ptr", "gemv_noalloc", "gemv_noalloc_ptr",
           "grouped_plane_shapes", "Status", "PnqError", "lib", "lib_path", "gemv", "dequantize_row", "validate_row",
           "quantize_row", "quantize_nvfp4_clip", "selftest_wait", "gemm", "gemm_scratch_bytes", "gemv_ptr", "dequantize_row_ptr", "validate_row_ptr", "quantize_row_ptr", "device_error",
           "nvfp4_weights", "pnq_grouped_weights"]
