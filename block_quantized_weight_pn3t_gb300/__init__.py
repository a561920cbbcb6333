"""pnq: block-quantized weight GEMV (pn3t, pn4t, NVFP4 W4A16) for sm_103a.

The compute path is the C-ABI library ``libpnq.so`` built from ``csrc/``; this
package only marshals arguments to it (see ``_binding``). Importing the package
does not load the library; the first call does, and raises if it is missing.
"""
from ._binding import (PN3T, PN4T, NVFP4, NVFP4_DIV, BLOCK_WEIGHTS, GEMV_STATIC_WEIGHTS, Status, PnqError, lib, lib_path, gemv,
                       gemv_ex_ptr, gemv_noalloc, gemv_noalloc_ptr,
                       dequantize_row, validate_row, gemv_ptr, dequantize_row_ptr, validate_row_ptr,
                       device_error, nvfp4_weights)

__all__ = ["PN3T", "PN4T", "NVFP4", "NVFP4_DIV", "BLOCK_WEIGHTS", "GEMV_STATIC_WEIGHTS", "gemv_ex_ptr", "gemv_noalloc",
           "gemv_noalloc_ptr", "Status", "PnqError", "lib", "lib_path", "gemv",
           "dequantize_row", "validate_row", "gemv_ptr", "dequantize_row_ptr", "validate_row_ptr",
           "device_error", "nvfp4_weights"]
