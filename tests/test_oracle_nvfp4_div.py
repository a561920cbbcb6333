"""Pins for the oracle's NVFP4 divisor reading ("tensor-formats.md" section 3.3: the global field
is one positive FP32 weight divisor d_w and W = decode_e2m1(c) * decode_e4m3fn(s) / d_w).

The decode is checked against the printed E2M1 grid (tests/golden) times torch's float8_e4m3fn
decode, divided by d_w in numpy float32 (an IEEE division, rounded once); special cases reduce it
to the multiplier reading (d_w = 1, d_w a power of two), and a planted multiplier fails. The GEMV
is checked against numpy's fp64 matmul of the same quotient and against a one-hot x.
"""
import numpy as np
import pytest
import torch

from golden_io import rows
from block_quantized_weight_pn3t_gb300 import synth


def grid():
    return {int(c, 16): float(v) for c, v in rows("e2m1_grid.txt")}


def torch_e4m3(s):
    return torch.from_numpy(np.ascontiguousarray(s)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def products(codes, scales, N, K):
    """e2m1 * e4m3 per weight, exact in float64 and in float32."""
    G = grid()
    nib = np.stack([codes & 15, codes >> 4], axis=-1).reshape(N, K)  # low nibble = even k
    e2 = np.vectorize(G.get)(nib).astype(np.float64)
    return e2 * np.repeat(torch_e4m3(scales), 16, axis=1)


@pytest.mark.parametrize("dw", [1.0, 3.0, 0.7, 2.0 ** -5, 448.0 * 6.0, 1.0e-30])
def test_dequant_div_matches_definition(oracle, dw):
    N, K = 20, 96
    codes, scales, _ = synth.nvfp4_random(N, K, seed=11)
    codes, scales = codes.numpy(), scales.numpy()
    prod = products(codes, scales, N, K)
    assert np.array_equal(prod.astype(np.float32).astype(np.float64), prod)  # the product is exact in fp32
    want = prod.astype(np.float32) / np.float32(dw)
    got = oracle.dequantize_nvfp4_div(codes, scales, float(dw), N, K)
    both_nan = np.isnan(want) & np.isnan(got)
    assert np.array_equal(got.view(np.uint32)[~both_nan], want.view(np.uint32)[~both_nan])


def test_unit_divisor_is_the_multiplier_decode(oracle):
    N, K = 16, 64
    codes, scales, _ = synth.nvfp4_random(N, K, seed=12)
    codes, scales = codes.numpy(), scales.numpy()
    a = oracle.dequantize_nvfp4_div(codes, scales, 1.0, N, K)
    b = oracle.dequantize_nvfp4(codes, scales, 1.0, N, K)
    nan = np.isnan(a)
    assert np.array_equal(nan, np.isnan(b)) and np.array_equal(a.view(np.uint32)[~nan], b.view(np.uint32)[~nan])


@pytest.mark.parametrize("k", [-7, -1, 3, 20])
def test_power_of_two_divisor_is_an_exact_multiplier(oracle, k):
    N, K = 8, 48
    codes, scales, _ = synth.nvfp4_random(N, K, seed=13 + k)
    codes, scales = codes.numpy(), scales.numpy()
    a = oracle.dequantize_nvfp4_div(codes, scales, 2.0 ** k, N, K)
    b = oracle.dequantize_nvfp4(codes, scales, 2.0 ** -k, N, K)
    nan = np.isnan(a)
    assert np.array_equal(a.view(np.uint32)[~nan], b.view(np.uint32)[~nan])


def test_a_multiplier_in_place_of_the_divisor_is_caught(oracle):
    """The pin above must tell the two readings apart: with d_w = 3 a multiplier decode differs."""
    N, K = 8, 32
    codes, scales, _ = synth.nvfp4_random(N, K, seed=14)
    codes, scales = codes.numpy(), scales.numpy()
    a = oracle.dequantize_nvfp4_div(codes, scales, 3.0, N, K)
    b = oracle.dequantize_nvfp4(codes, scales, 3.0, N, K)
    finite = np.isfinite(a) & (a != 0)
    assert finite.any() and not np.array_equal(a[finite], b[finite])


@pytest.mark.parametrize("dw", [0.37, 5.0e3])
def test_gemv_div_against_fp64_matmul(oracle, dw):
    N, K, M = 33, 128, 3
    codes, scales, _ = synth.nvfp4_random(N, K, seed=15)
    codes, scales = codes.numpy(), scales.numpy()
    Xb = synth.activations_bf16(M, K, seed=16)
    x = (Xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    W = products(codes, scales, N, K) / np.float64(np.float32(dw))
    Y, A = oracle.gemv_nvfp4_div(codes, scales, float(dw), N, K, Xb)
    ok = np.isfinite(W).all(axis=1)
    ref = x @ W[ok].T
    aref = np.abs(x) @ np.abs(W[ok]).T
    assert np.all(np.abs(Y[:, ok] - ref) <= 1e-12 * aref)
    assert np.allclose(A[:, ok], aref, rtol=1e-12)


def test_gemv_div_one_hot_is_the_quotient(oracle):
    N, K, dw = 12, 64, 0.3
    codes, scales, _ = synth.nvfp4_random(N, K, seed=17)
    codes, scales = codes.numpy(), scales.numpy()
    W = products(codes, scales, N, K) / np.float64(np.float32(dw))
    for k in (0, 17, 63):
        Xb = np.zeros((1, K), dtype=np.uint16)
        Xb[0, k] = 0x3F80  # bf16 1.0
        Y, _ = oracle.gemv_nvfp4_div(codes, scales, dw, N, K, Xb)
        ok = np.isfinite(W[:, k])
        assert np.array_equal(Y[0, ok], W[ok, k])
