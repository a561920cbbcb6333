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
Q4G64, Q5G64, Q6G64, W8G32 = 1104, 1105, 1106, 1108
GROUPED = {Q4G64: (4, 64, -8, 7), Q5G64: (5, 64, -16, 15), Q6G64: (6, 64, -32, 31), W8G32: (8, 32, -127, 127)}
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
            "pnq_ref_dequantize_row_nvfp4_div": (I32, [P, P, F, I64, I64, P]),
            "pnq_ref_grouped_plane_bytes": (I32, [I32, I64, P, P, P]),
            "pnq_ref_dequantize_grouped": (I32, [I32, P, P, P, I64, I64, P]),
            "pnq_ref_validate_grouped": (I32, [I32, P, P, P, I64, I64, P]),
            "pnq_ref_quantize_grouped": (I32, [I32, P, I64, I64, P, P, P, P]),
            "pnq_ref_gemv_grouped": (I32, [I32, P, P, P, I64, I64, P, I32, P, P]),
            "pnq_ref_quantize_nvfp4_clip": (I32, [P, P, F, I64, I64, P, P, P]),
            "pnq_ref_gemv_nvfp4_div": (I32, [P, P, F, I64, I64, P, I32, P, P]),
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


def dequantize_nvfp4_div(codes: np.ndarray, scales: np.ndarray, dw: float, n_rows: int, K: int) -> np.ndarray:
    """NVFP4 with the global field as a divisor: fp32(e2m1 * e4m3) / d_w."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    out = np.empty((n_rows, K), dtype=np.float32)
    _check(lib().pnq_ref_dequantize_row_nvfp4_div(_ptr(codes), _ptr(scales), dw, n_rows, K, _ptr(out)),
           "dequantize_nvfp4_div")
    return out


def gemv_nvfp4_div(codes: np.ndarray, scales: np.ndarray, dw: float, N: int, K: int, X_bf16: np.ndarray):
    """X_bf16: uint16 [M][K] raw bf16 words; the weight is e2m1 * e4m3 / d_w."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    X = np.ascontiguousarray(X_bf16, dtype=np.uint16)
    if X.ndim == 1:
        X = X[None, :]
    M = X.shape[0]
    Y = np.empty((M, N), dtype=np.float64)
    A = np.empty((M, N), dtype=np.float64)
    _check(lib().pnq_ref_gemv_nvfp4_div(_ptr(codes), _ptr(scales), dw, N, K, _ptr(X), M, _ptr(Y), _ptr(A)),
           "gemv_nvfp4_div")
    return Y, A


# ---- grouped signed-integer formats ("tensor-formats.md" sections 4 to 7) ----

def grouped_plane_bytes(type_: int, K: int):
    """(lo bytes, hi bytes, scales) per row of the library's plane layout."""
    lo, hi, ns = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _check(lib().pnq_ref_grouped_plane_bytes(type_, K, ctypes.byref(lo), ctypes.byref(hi), ctypes.byref(ns)),
           "grouped_plane_bytes")
    return lo.value, hi.value, ns.value


def _planes(type_, lo, hi, sc):
    lo = np.ascontiguousarray(lo, dtype=np.uint8)
    hi = None if hi is None else np.ascontiguousarray(hi, dtype=np.uint8)
    sc = np.ascontiguousarray(sc, dtype=np.uint16)
    return lo, hi, sc


def dequantize_grouped(type_: int, lo, hi, sc, n_rows: int, K: int) -> np.ndarray:
    lo, hi, sc = _planes(type_, lo, hi, sc)
    out = np.empty((n_rows, K), dtype=np.float32)
    _check(lib().pnq_ref_dequantize_grouped(type_, _ptr(lo), None if hi is None else _ptr(hi), _ptr(sc), n_rows, K,
                                            _ptr(out)), "dequantize_grouped")
    return out


def validate_grouped(type_: int, lo, hi, sc, n_rows: int, K: int) -> np.ndarray:
    lo, hi, sc = _planes(type_, lo, hi, sc)
    flags = np.empty(n_rows, dtype=np.int32)
    _check(lib().pnq_ref_validate_grouped(type_, _ptr(lo), None if hi is None else _ptr(hi), _ptr(sc), n_rows, K,
                                          _ptr(flags)), "validate_grouped")
    return flags


def quantize_grouped(type_: int, w: np.ndarray):
    """Canonical encoder MAXABS_F16_RECIP_RNE_V1 on a [n_rows][K] float32 matrix. Returns
    (lo, hi or None, scales); ValueError for a group the profile rejects (non-finite value or
    an overflowing scale)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    n_rows, K = w.shape
    lb, hb, ns = grouped_plane_bytes(type_, K)
    lo = np.zeros((n_rows, lb), dtype=np.uint8)
    hi = np.zeros((n_rows, hb), dtype=np.uint8) if hb else None
    sc = np.zeros((n_rows, ns), dtype=np.uint16)
    fail = ctypes.c_int64(-1)
    _check(lib().pnq_ref_quantize_grouped(type_, _ptr(w), n_rows, K, _ptr(lo), None if hi is None else _ptr(hi),
                                          _ptr(sc), ctypes.byref(fail)), "quantize_grouped")
    return lo, hi, sc


def gemv_grouped(type_: int, lo, hi, sc, N: int, K: int, X: np.ndarray):
    lo, hi, sc = _planes(type_, lo, hi, sc)
    X = np.ascontiguousarray(X, dtype=np.float32)
    if X.ndim == 1:
        X = X[None, :]
    M = X.shape[0]
    Y = np.empty((M, N), dtype=np.float64)
    A = np.empty((M, N), dtype=np.float64)
    _check(lib().pnq_ref_gemv_grouped(type_, _ptr(lo), None if hi is None else _ptr(hi), _ptr(sc), N, K, _ptr(X), M,
                                      _ptr(Y), _ptr(A)), "gemv_grouped")
    return Y, A


def quantize_nvfp4_clip(w: np.ndarray, act_ms: np.ndarray, g: float):
    """NVFP4 clip search on a [N][K] fp32 matrix with per-channel act_ms [K]; returns
    (codes [N][K/2], scales [N][K/16], chosen multiplier index [N][K/16])."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    act_ms = np.ascontiguousarray(act_ms, dtype=np.float32)
    N, K = w.shape
    codes = np.empty((N, K // 2), dtype=np.uint8)
    scales = np.empty((N, K // 16), dtype=np.uint8)
    chosen = np.empty((N, K // 16), dtype=np.int32)
    _check(lib().pnq_ref_quantize_nvfp4_clip(_ptr(w), _ptr(act_ms), g, N, K, _ptr(codes), _ptr(scales), _ptr(chosen)),
           "quantize_nvfp4_clip")
    return codes, scales, chosen
