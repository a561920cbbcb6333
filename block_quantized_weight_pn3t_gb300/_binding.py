"""Thin ctypes binding to libpnq.so: argument marshalling only, same names as the C ABI.

Every computation runs in the library's CUDA kernels. There is no fallback: if the
library is missing or fails to load, the first call raises ``PnqError``.
"""
from __future__ import annotations

import ctypes
import enum
import os

PN3T, PN4T, NVFP4, NVFP4_DIV = 124, 125, 1004, 1005
Q4G64_F16S, Q5G64_F16S, Q6G64_F16S, W8G32_F16S = 1104, 1105, 1106, 1108
NVFP4_TYPES = (NVFP4, NVFP4_DIV)
BLOCK_WEIGHTS = {PN3T: 80, PN4T: 64}
# grouped signed-integer formats: (code bits, group size)
GROUPED = {Q4G64_F16S: (4, 64), Q5G64_F16S: (5, 64), Q6G64_F16S: (6, 64), W8G32_F16S: (8, 32)}


def grouped_plane_shapes(type_: int, n_rows: int, K: int):
    """Shapes of the (lo, hi, scales) planes of an [n_rows][K] grouped matrix (hi None for Q4, W8)."""
    bits, G = GROUPED[type_]
    lo = (n_rows, K if bits == 8 else K // 2)
    hi = {5: (n_rows, K // 8), 6: (n_rows, K // 4)}.get(bits)
    return lo, hi, (n_rows, (K + G - 1) // G)

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libpnq.so")


class Status(enum.IntEnum):
    OK = 0
    ERR_TYPE = -1
    ERR_SHAPE = -2
    ERR_NULL = -3
    ERR_ALIGN = -4
    ERR_CUDA = -5
    ERR_DEVICE = -6
    ERR_FLAGS = -7
    ERR_SCRATCH = -8
    ERR_VALUE = -9


GEMV_STATIC_WEIGHTS = 1


class PnqError(RuntimeError):
    def __init__(self, what: str, status: int | None = None):
        self.status = status
        super().__init__(what if status is None else f"{what}: {Status(status).name} ({status})")


class pnq_nvfp4_weights(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("global_scale", ctypes.c_float)]


class pnq_grouped_weights(ctypes.Structure):
    _fields_ = [("lo", ctypes.c_void_p), ("hi", ctypes.c_void_p), ("scales", ctypes.c_void_p)]


_lib = None


def lib_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """Load libpnq.so (built by ``__graft_entry__.build()``); raise if it is not there."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise PnqError(f"{_LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
        try:
            L = ctypes.CDLL(_LIB_PATH)
        except OSError as e:
            raise PnqError(f"cannot load {_LIB_PATH}: {e}") from e
        P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.pnq_gemv.restype = I
        L.pnq_gemv.argtypes = [I, P, I64, I64, P, I, P, P]
        L.pnq_gemv_ex.restype = I
        L.pnq_gemv_ex.argtypes = [I, P, I64, I64, P, I, P, ctypes.c_uint, P]
        L.pnq_gemv_noalloc.restype = I
        L.pnq_gemv_noalloc.argtypes = [I, P, I64, I64, P, I, P, ctypes.c_uint, P]
        L.pnq_dequantize_row.restype = I
        L.pnq_dequantize_row.argtypes = [I, P, I64, I64, P, P]
        L.pnq_validate_row.restype = I
        L.pnq_validate_row.argtypes = [I, P, I64, I64, P, P]
        L.pnq_quantize_row.restype = I
        L.pnq_quantize_row.argtypes = [I, P, I64, I64, P, P, P]
        L.pnq_quantize_nvfp4_clip.restype = I
        L.pnq_quantize_nvfp4_clip.argtypes = [P, P, I64, I64, ctypes.c_float, P, P, P, P]
        L.pnq_selftest_wait.restype = I
        L.pnq_selftest_wait.argtypes = [ctypes.c_uint32, P]
        L.pnq_gemm.restype = I
        L.pnq_gemm.argtypes = [I, P, I64, I64, P, I64, P, P, ctypes.c_uint64, P]
        L.pnq_gemm_scratch_bytes.restype = I
        L.pnq_gemm_scratch_bytes.argtypes = [I, I64, I64, I64, I64, ctypes.POINTER(ctypes.c_uint64)]
        L.pnq_device_error.restype = I
        L.pnq_device_error.argtypes = [ctypes.POINTER(ctypes.c_int32)]
        L.pnq_version.restype = ctypes.c_char_p
        L.pnq_version.argtypes = []
        _lib = L
    return _lib


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise PnqError(what, rc)


def nvfp4_weights(codes_ptr: int, scales_ptr: int, global_scale: float) -> pnq_nvfp4_weights:
    return pnq_nvfp4_weights(codes_ptr, scales_ptr, float(global_scale))


def _w_arg(type_: int, W):
    """PN: W is a device address (int). NVFP4: W is a pnq_nvfp4_weights (passed by host pointer)."""
    if type_ in NVFP4_TYPES:
        if not isinstance(W, pnq_nvfp4_weights):
            raise TypeError("NVFP4 weights must be a pnq_nvfp4_weights descriptor")
        return ctypes.byref(W)
    if type_ in GROUPED:
        if not isinstance(W, pnq_grouped_weights):
            raise TypeError("grouped weights must be a pnq_grouped_weights descriptor")
        return ctypes.byref(W)
    return ctypes.c_void_p(W)


# ---- raw entry points (integer addresses; stream as an integer handle) ----------------

def gemv_ptr(type_: int, W, N: int, K: int, X: int, M: int, Y: int, stream: int = 0) -> int:
    return lib().pnq_gemv(type_, _w_arg(type_, W), N, K, ctypes.c_void_p(X), M, ctypes.c_void_p(Y),
                          ctypes.c_void_p(stream))


def gemv_ex_ptr(type_: int, W, N: int, K: int, X: int, M: int, Y: int, flags: int, stream: int = 0) -> int:
    return lib().pnq_gemv_ex(type_, _w_arg(type_, W), N, K, ctypes.c_void_p(X), M, ctypes.c_void_p(Y),
                             flags, ctypes.c_void_p(stream))


def gemv_noalloc_ptr(type_: int, W, N: int, K: int, X: int, M: int, Y: int, flags: int = 0, stream: int = 0) -> int:
    return lib().pnq_gemv_noalloc(type_, _w_arg(type_, W), N, K, ctypes.c_void_p(X), M, ctypes.c_void_p(Y),
                                  flags, ctypes.c_void_p(stream))


def dequantize_row_ptr(type_: int, W, n_rows: int, K: int, out: int, stream: int = 0) -> int:
    return lib().pnq_dequantize_row(type_, _w_arg(type_, W), n_rows, K, ctypes.c_void_p(out),
                                    ctypes.c_void_p(stream))


def validate_row_ptr(type_: int, W, n_rows: int, K: int, flags: int, stream: int = 0) -> int:
    return lib().pnq_validate_row(type_, _w_arg(type_, W), n_rows, K, ctypes.c_void_p(flags),
                                  ctypes.c_void_p(stream))


def quantize_row_ptr(type_: int, w: int, n_rows: int, K: int, out, status: int, stream: int = 0) -> int:
    """out: a device address (PN) or a pnq_grouped_weights holding the output planes (grouped)."""
    o = ctypes.byref(out) if type_ in GROUPED else ctypes.c_void_p(out)
    return lib().pnq_quantize_row(type_, ctypes.c_void_p(w), n_rows, K, o, ctypes.c_void_p(status),
                                  ctypes.c_void_p(stream))


def selftest_wait(limit_us: int, stream=None) -> None:
    """Run the bounded-wait self-test (a wait nothing completes, giving up after limit_us)."""
    _check(lib().pnq_selftest_wait(int(limit_us), ctypes.c_void_p(_stream_handle(stream) if stream is not None else 0)),
           "pnq_selftest_wait")


def device_error() -> int:
    code = ctypes.c_int32(0)
    rc = lib().pnq_device_error(ctypes.byref(code))
    if rc not in (0, int(Status.ERR_DEVICE)):
        raise PnqError("pnq_device_error", rc)
    return int(code.value)


# ---- torch tensor wrappers (marshalling only) ----------------------------------------------

def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _require(t, what: str, dtypes, numel: int | None = None) -> None:
    """Raise PnqError unless t is a contiguous CUDA tensor of one of `dtypes` holding at least
    `numel` elements (the library receives only its address)."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise PnqError(f"{what} must be a torch.Tensor, not {type(t).__name__}")
    if t.dtype not in dtypes:
        raise PnqError(f"{what} has dtype {t.dtype}; expected {' or '.join(str(d) for d in dtypes)}")
    if not t.is_contiguous():
        raise PnqError(f"{what} must be contiguous")
    if numel is not None and t.numel() < numel:
        raise PnqError(f"{what} holds {t.numel()} elements; the call needs {numel}")
    if not t.is_cuda:
        raise PnqError(f"{what} must be a CUDA tensor (device {t.device})")


def _check_weights(type_: int, W, n_rows: int, K: int) -> None:
    import torch
    if type_ in NVFP4_TYPES:
        codes, scales, _g = W
        whole = K > 0 and K % 16 == 0
        _require(codes, "NVFP4 codes", (torch.uint8,), n_rows * K // 2 if whole else None)
        _require(scales, "NVFP4 scales", (torch.uint8,), n_rows * K // 16 if whole else None)
    elif type_ in BLOCK_WEIGHTS:
        blk = BLOCK_WEIGHTS[type_]
        _require(W, "W", (torch.uint8,), n_rows * (K // blk) * 34 if K > 0 and K % blk == 0 else None)
    elif type_ in GROUPED:
        lo, hi, sc = W
        shapes = grouped_plane_shapes(type_, n_rows, K) if K > 0 and K % 8 == 0 else (None, None, None)
        _require(lo, "grouped lo plane", (torch.uint8, torch.int8), None if shapes[0] is None else shapes[0][0] * shapes[0][1])
        if shapes[1] is not None:
            _require(hi, "grouped hi plane", (torch.uint8,), shapes[1][0] * shapes[1][1])
        _require(sc, "grouped scales", (torch.uint16, torch.int16, torch.float16),
                 None if shapes[2] is None else shapes[2][0] * shapes[2][1])
    # an unknown type is left to the library (PNQ_ERR_TYPE)


def _check_x(type_: int, X, K: int) -> int:
    """The activation rows M of X ([M][K], or [K] for M = 1), after checking X."""
    import torch
    dtypes = (torch.bfloat16, torch.int16) if type_ in NVFP4_TYPES else (torch.float32,)  # PN, grouped: fp32
    M = X.shape[0] if X.dim() == 2 else 1
    _require(X, "X", dtypes)
    if X.numel() != M * K:
        raise PnqError(f"X has shape {tuple(X.shape)}; expected [M][{K}] or [{K}]")
    return M


def _weights(type_: int, W):
    if type_ in NVFP4_TYPES:
        codes, scales, g = W
        return nvfp4_weights(codes.data_ptr(), scales.data_ptr(), g)
    if type_ in GROUPED:
        lo, hi, sc = W
        return pnq_grouped_weights(lo.data_ptr(), 0 if hi is None else hi.data_ptr(), sc.data_ptr())
    return W.data_ptr()


def gemv(type_: int, W, X, N: int, K: int, Y=None, stream=None, flags: int = 0):
    """Y[m][n] = sum_k W[n][k] X[m][k]. W: uint8 CUDA tensor of PN blocks, or (codes, scales, g)
    for NVFP4. X: CUDA [M][K] fp32 (PN) or bf16 (NVFP4). Returns Y (CUDA fp32 [M][N])."""
    import torch
    _check_weights(type_, W, N, K)
    M = _check_x(type_, X, K)
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float32, device=X.device)
    _require(Y, "Y", (torch.float32,), M * N)
    _check(gemv_ex_ptr(type_, _weights(type_, W), N, K, X.data_ptr(), M, Y.data_ptr(), flags,
                       _stream_handle(stream)), "pnq_gemv_ex")
    return Y


def gemv_noalloc(type_: int, W, X, N: int, K: int, Y=None, stream=None, flags: int = 0):
    """gemv through pnq_gemv_noalloc (no device allocation; PnqError ERR_SCRATCH when the shape
    needs more than the library's built-in scratch)."""
    import torch
    _check_weights(type_, W, N, K)
    M = _check_x(type_, X, K)
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float32, device=X.device)
    _require(Y, "Y", (torch.float32,), M * N)
    _check(gemv_noalloc_ptr(type_, _weights(type_, W), N, K, X.data_ptr(), M, Y.data_ptr(), flags,
                            _stream_handle(stream)), "pnq_gemv_noalloc")
    return Y


def dequantize_row(type_: int, W, n_rows: int, K: int, out=None, stream=None):
    import torch
    _check_weights(type_, W, n_rows, K)
    if out is None:
        dev = W[0].device if isinstance(W, tuple) else W.device
        out = torch.empty((n_rows, K), dtype=torch.float32, device=dev)
    _require(out, "out", (torch.float32,), n_rows * K)
    _check(dequantize_row_ptr(type_, _weights(type_, W), n_rows, K, out.data_ptr(), _stream_handle(stream)),
           "pnq_dequantize_row")
    return out


def validate_row(type_: int, W, n_rows: int, K: int, flags=None, stream=None):
    import torch
    _check_weights(type_, W, n_rows, K)
    if flags is None:
        dev = W[0].device if isinstance(W, tuple) else W.device
        flags = torch.empty((n_rows,), dtype=torch.int32, device=dev)
    _require(flags, "flags", (torch.int32,), n_rows)
    _check(validate_row_ptr(type_, _weights(type_, W), n_rows, K, flags.data_ptr(), _stream_handle(stream)),
           "pnq_validate_row")
    return flags


def quantize_row(type_: int, w, out=None, status=None, stream=None):
    """Encode a CUDA fp32 [n_rows][K] matrix on the GPU: the PN reference quantizer (returns the
    uint8 blocks) or the grouped canonical encoder (returns (lo, hi or None, scales)); also
    returns the per-row status (int32, 1 = row rejected)."""
    import torch
    _require(w, "w", (torch.float32,))
    if w.dim() != 2:
        raise PnqError(f"w has shape {tuple(w.shape)}; expected [n_rows][K]")
    n_rows, K = w.shape
    if status is None:
        status = torch.empty((n_rows,), dtype=torch.int32, device=w.device)
    _require(status, "status", (torch.int32,), n_rows)
    if type_ in GROUPED:
        if out is None:
            slo, shi, ssc = grouped_plane_shapes(type_, n_rows, K)
            out = (torch.empty(slo, dtype=torch.uint8, device=w.device),
                   None if shi is None else torch.empty(shi, dtype=torch.uint8, device=w.device),
                   torch.empty(ssc, dtype=torch.int16, device=w.device))
        desc = pnq_grouped_weights(out[0].data_ptr(), 0 if out[1] is None else out[1].data_ptr(), out[2].data_ptr())
        _check(quantize_row_ptr(type_, w.data_ptr(), n_rows, K, desc, status.data_ptr(), _stream_handle(stream)),
               "pnq_quantize_row")
        return out, status
    if out is None:
        blk = BLOCK_WEIGHTS.get(type_, 1)
        out = torch.empty((n_rows * (K // blk) * 34,), dtype=torch.uint8, device=w.device)
    _require(out, "out", (torch.uint8,))
    _check(quantize_row_ptr(type_, w.data_ptr(), n_rows, K, out.data_ptr(), status.data_ptr(), _stream_handle(stream)),
           "pnq_quantize_row")
    return out, status


def quantize_nvfp4_clip(w, act_ms, global_scale: float, stream=None):
    """NVFP4 clip search on the GPU: w CUDA fp32 [n_rows][K], act_ms CUDA fp32 [K]. Returns
    (codes uint8 [n_rows][K/2], scales uint8 [n_rows][K/16], row status int32 [n_rows])."""
    import torch
    _require(w, "w", (torch.float32,))
    if w.dim() != 2:
        raise PnqError(f"w has shape {tuple(w.shape)}; expected [n_rows][K]")
    n_rows, K = w.shape
    _require(act_ms, "act_ms", (torch.float32,), K)
    codes = torch.empty((n_rows, K // 2), dtype=torch.uint8, device=w.device)
    scales = torch.empty((n_rows, max(K // 16, 0)), dtype=torch.uint8, device=w.device)
    status = torch.empty((n_rows,), dtype=torch.int32, device=w.device)
    _check(lib().pnq_quantize_nvfp4_clip(ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(act_ms.data_ptr()), n_rows, K,
                                         float(global_scale), ctypes.c_void_p(codes.data_ptr()),
                                         ctypes.c_void_p(scales.data_ptr()), ctypes.c_void_p(status.data_ptr()),
                                         ctypes.c_void_p(_stream_handle(stream))), "pnq_quantize_nvfp4_clip")
    return codes, scales, status


def gemm_scratch_bytes(type_: int, N: int, K: int, M: int, slice_rows: int = 0) -> int:
    out = ctypes.c_uint64(0)
    _check(lib().pnq_gemm_scratch_bytes(type_, N, K, M, slice_rows, ctypes.byref(out)), "pnq_gemm_scratch_bytes")
    return int(out.value)


def gemm(type_: int, W, X, N: int, K: int, Y=None, scratch=None, slice_rows: int = 0, stream=None):
    """Y[m][n] = sum_k W[n][k] X[m][k] for any M (prefill path, PN types). W: uint8 CUDA tensor of PN
    blocks; X: CUDA fp32 [M][K]. scratch: a CUDA uint8 tensor of at least
    gemm_scratch_bytes(type_, N, K, M, slice_rows) bytes (made here when None)."""
    import torch
    _check_weights(type_, W, N, K)
    _require(X, "X", (torch.float32,))
    M = X.shape[0] if X.dim() == 2 else 1
    if X.numel() != M * K:
        raise PnqError(f"X has shape {tuple(X.shape)}; expected [M][{K}]")
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float32, device=X.device)
    _require(Y, "Y", (torch.float32,), M * N)
    if scratch is None:
        scratch = torch.empty((gemm_scratch_bytes(type_, N, K, M, slice_rows),), dtype=torch.uint8, device=X.device)
    _require(scratch, "scratch", (torch.uint8,))
    _check(lib().pnq_gemm(type_, ctypes.c_void_p(W.data_ptr()), N, K, ctypes.c_void_p(X.data_ptr()), M,
                          ctypes.c_void_p(Y.data_ptr()), ctypes.c_void_p(scratch.data_ptr()), scratch.numel(),
                          ctypes.c_void_p(_stream_handle(stream))), "pnq_gemm")
    return Y
