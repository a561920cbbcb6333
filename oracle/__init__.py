"""ctypes binding for the CPU oracle in ``pnq_oracle.c``.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT. Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import this package. It shares no code with the CUDA library
in ``block_quantized_weight_pn3t_gb300``; see ``pnq_oracle.h`` for what each
routine restates from the format pages.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pnq_oracle.c")
LIB_PATH = os.path.join(_HERE, "libpnq_oracle.so")

PN3T, PN4T, NVFP4 = 124, 125, 1004
BLOCK_WEIGHTS = {PN3T: 80, PN4T: 64}
OK = 0


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (plain -O2, no fast-math)."""
    stale = (not os.path.exists(LIB_PATH)
             or os.path.getmtime(LIB_PATH) < max(os.path.getmtime(_SRC),
                                                 os.path.getmtime(os.path.join(_HERE, "pnq_oracle.h"))))
    if force or stale:
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fno-fast-math", "-ffp-contract=off",
                               "-Wall", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


_lib = None


def lib() -> ctypes.CDLL:
    """The oracle library, built on first use. PNQ_ORACLE_LIB names another build of the same
    source to load instead (the mutation tests load copies with a planted mistake)."""
    global _lib
    if _lib is None:
        path = os.environ.get("PNQ_ORACLE_LIB") or build()
        L = ctypes.CDLL(path)
        P, I64, I32, F, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_double
        sig = {
            "pnq_ref_block_weights": (I32, [I32]),
            "pnq_ref_fp16_to_double": (D, [ctypes.c_uint16]),
            "pnq_ref_double_to_fp16": (ctypes.c_uint16, [D]),
            "pnq_ref_bf16_to_double": (D, [ctypes.c_uint16]),
            "pnq_ref_e2m1_to_double": (D, [ctypes.c_uint8]),
            "pnq_ref_e4m3fn_to_double": (D, [ctypes.c_uint8]),
            "pnq_ref_dequantize_row": (I32, [I32, P, I64, I64, P]),
            "pnq_ref_dequantize_row_elemshift": (I32, [I32, P, I64, I64, P]),
            "pnq_ref_validate_row": (I32, [I32, P, I64, I64, P]),
            "pnq_ref_quantize_row": (I32, [I32, P, I64, P, P]),
            "pnq_ref_dequantize_row_nvfp4": (I32, [P, P, F, I64, I64, P]),
            "pnq_ref_validate_row_nvfp4": (I32, [P, F, I64, I64, P]),
            "pnq_ref_gemv": (I32, [I32, P, I64, I64, P, I32, P, P]),
            "pnq_ref_gemv_nvfp4": (I32, [P, P, F, I64, I64, P, I32, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype, fn.argtypes = res, args
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _check(rc: int, what: str) -> None:
    if rc != OK:
        raise ValueError(f"{what} failed with status {rc}")


def row_bytes(type_: int, K: int) -> int:
    return (K // BLOCK_WEIGHTS[type_]) * 34


# ---- scalar codecs -----------------------------------------------------------

def fp16_to_double(h: int) -> float:
    return lib().pnq_ref_fp16_to_double(h)


def double_to_fp16(x: float) -> int:
    return lib().pnq_ref_double_to_fp16(x)


def bf16_to_double(b: int) -> float:
    return lib().pnq_ref_bf16_to_double(b)


def e2m1_to_double(c: int) -> float:
    return lib().pnq_ref_e2m1_to_double(c)


def e4m3fn_to_double(c: int) -> float:
    return lib().pnq_ref_e4m3fn_to_double(c)


# ---- PN --------------------------------------------------------------------------

def dequantize(type_: int, W: np.ndarray, n_rows: int, K: int) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.uint8)
    assert W.size >= n_rows * row_bytes(type_, K)
    out = np.empty((n_rows, K), dtype=np.float32)
    _check(lib().pnq_ref_dequantize_row(type_, _ptr(W), n_rows, K, _ptr(out)), "dequantize")
    return out


def dequantize_elemshift(type_: int, W: np.ndarray, n_rows: int, K: int) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.uint8)
    out = np.empty((n_rows, K), dtype=np.float32)
    _check(lib().pnq_ref_dequantize_row_elemshift(type_, _ptr(W), n_rows, K, _ptr(out)), "elemshift")
    return out


def validate(type_: int, W: np.ndarray, n_rows: int, K: int) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.uint8)
    flags = np.empty(n_rows, dtype=np.int32)
    _check(lib().pnq_ref_validate_row(type_, _ptr(W), n_rows, K, _ptr(flags)), "validate")
    return flags


def quantize(type_: int, w: np.ndarray, return_m: bool = False):
    """Quantize a 2-D fp32 matrix [N][K] row by row; returns uint8 [N][row_bytes]."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    if w.ndim == 1:
        w = w[None, :]
    N, K = w.shape
    nb = K // BLOCK_WEIGHTS[type_]
    out = np.empty((N, nb * 34), dtype=np.uint8)
    ms = np.empty((N, nb), dtype=np.float64)
    for n in range(N):
        row_out = out[n]
        row_m = ms[n]
        _check(lib().pnq_ref_quantize_row(type_, _ptr(w[n]), K, row_out.ctypes.data, row_m.ctypes.data),
               "quantize")
    return (out, ms) if return_m else out


def gemv(type_: int, W: np.ndarray, N: int, K: int, X: np.ndarray):
    """fp64 (Y, A) with Y[m][n] = sum_k w[n][k] x[m][k] and A the sum of |w x|."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    X = np.ascontiguousarray(X, dtype=np.float32)
    if X.ndim == 1:
        X = X[None, :]
    M = X.shape[0]
    assert X.shape[1] == K
    Y = np.empty((M, N), dtype=np.float64)
    A = np.empty((M, N), dtype=np.float64)
    _check(lib().pnq_ref_gemv(type_, _ptr(W), N, K, _ptr(X), M, _ptr(Y), _ptr(A)), "gemv")
    return Y, A


# ---- NVFP4 ---------------------------------------------------------------------------

def dequantize_nvfp4(codes: np.ndarray, scales: np.ndarray, g: float, n_rows: int, K: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    out = np.empty((n_rows, K), dtype=np.float32)
    _check(lib().pnq_ref_dequantize_row_nvfp4(_ptr(codes), _ptr(scales), g, n_rows, K, _ptr(out)),
           "dequantize_nvfp4")
    return out


def validate_nvfp4(scales: np.ndarray, g: float, n_rows: int, K: int) -> np.ndarray:
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    flags = np.empty(n_rows, dtype=np.int32)
    _check(lib().pnq_ref_validate_row_nvfp4(_ptr(scales), g, n_rows, K, _ptr(flags)), "validate_nvfp4")
    return flags


def gemv_nvfp4(codes: np.ndarray, scales: np.ndarray, g: float, N: int, K: int, X_bf16: np.ndarray):
    """X_bf16: uint16 [M][K] raw bf16 words."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    X = np.ascontiguousarray(X_bf16, dtype=np.uint16)
    if X.ndim == 1:
        X = X[None, :]
    M = X.shape[0]
    Y = np.empty((M, N), dtype=np.float64)
    A = np.empty((M, N), dtype=np.float64)
    _check(lib().pnq_ref_gemv_nvfp4(_ptr(codes), _ptr(scales), g, N, K, _ptr(X), M, _ptr(Y), _ptr(A)),
           "gemv_nvfp4")
    return Y, A
