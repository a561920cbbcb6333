"""Pins for the oracle's NVFP4 decode / validation and for both GEMV oracles.

NVFP4 weights are checked against the printed E2M1 grid (tests/golden) times torch's
float8_e4m3fn decode times the global multiplier. The GEMVs are checked against closed
forms (one-hot x gives a dequantized column exactly; constant codes give d*(n-z)*K) and
against numpy's matmul of the dequantized matrix in fp64.
"""
import numpy as np
import pytest
import torch

from golden_io import rows
from block_quantized_weight_pn3t_gb300 import synth

PN3T, PN4T = 124, 125
BLK = {PN3T: 80, PN4T: 64}


def grid():
    return {int(c, 16): float(v) for c, v in rows("e2m1_grid.txt")}


def torch_e4m3(s):
    return torch.from_numpy(np.ascontiguousarray(s)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_nvfp4_dequant_matches_definition(oracle):
    N, K = 24, 64
    codes, scales, g = synth.nvfp4_random(N, K, seed=4)
    codes, scales = codes.numpy(), scales.numpy()
    g = np.float32(0.01)
    out = oracle.dequantize_nvfp4(codes, scales, float(g), N, K)
    G = grid()
    nib = np.stack([codes & 15, codes >> 4], axis=-1).reshape(N, K)  # low nibble = even k
    e2 = np.vectorize(G.get)(nib).astype(np.float64)
    sc = np.repeat(torch_e4m3(scales), 16, axis=1)
    want = (e2 * sc * np.float64(g)).astype(np.float32)
    assert np.array_equal(out.view(np.uint32), want.view(np.uint32))


def test_nvfp4_dequant_all_code_scale_pairs(oracle):
    """Every (code, scale) pair: exact product e2m1 * e4m3, then one rounding with g."""
    G = grid()
    codes = np.zeros((256, 8), dtype=np.uint8)
    scales = np.zeros((256, 1), dtype=np.uint8)
    for s in range(256):
        scales[s, 0] = s
        codes[s] = [(2 * i) | ((2 * i + 1) << 4) for i in range(8)]  # codes 0..15 in order
    for g in (1.0, 0.01, 3.0e-5):
        out = oracle.dequantize_nvfp4(codes, scales, g, 256, 16)
        sc = torch_e4m3(scales[:, 0])
        for s in range(256):
            for c in range(16):
                want = np.float32(G[c] * sc[s] * np.float64(np.float32(g)))
                got = out[s, c]
                if np.isnan(want):
                    assert np.isnan(got)
                else:
                    assert got == want and np.signbit(got) == np.signbit(want), (s, c, g)


def test_nvfp4_validate(oracle):
    N, K = 10, 32
    scales = np.full((N, K // 16), 0x38, dtype=np.uint8)  # 1.0
    want = [0] * N
    for r, bad in ((1, 0x80), (2, 0xB8), (3, 0x7F), (4, 0xFF)):
        scales[r, 1] = bad
        want[r] = 1
    for r, ok in ((5, 0x00), (6, 0x7E), (7, 0x01)):
        scales[r, 0] = ok
    assert oracle.validate_nvfp4(scales, 0.01, N, K).tolist() == want
    for g in (0.0, -1.0, float("inf"), float("nan")):
        assert oracle.validate_nvfp4(scales, g, N, K).tolist() == [1] * N


@pytest.mark.parametrize("type_", [PN3T, PN4T])
def test_pn_gemv_vs_numpy_and_one_hot(oracle, type_):
    N, K, M = 40, BLK[type_] * 8, 3
    W = synth.pn_random_blocks(type_, N, K, seed=8).numpy()
    X = synth.activations(M, K, seed=8)
    Y, A = oracle.gemv(type_, W, N, K, X)
    Wd = oracle.dequantize(type_, W, N, K).astype(np.float64)
    ref = X.astype(np.float64) @ Wd.T
    assert np.allclose(Y, ref, rtol=1e-12, atol=1e-15)
    assert np.allclose(A, np.abs(X.astype(np.float64)) @ np.abs(Wd).T, rtol=1e-12, atol=1e-15)
    assert np.all(A >= np.abs(Y))
    for k in (0, 1, BLK[type_] - 1, BLK[type_], K - 1):
        onehot = np.zeros((1, K), dtype=np.float32)
        onehot[0, k] = 1.0
        Y1, _ = oracle.gemv(type_, W, N, K, onehot)
        assert np.array_equal(Y1[0], Wd[:, k])
    Y0, A0 = oracle.gemv(type_, W, N, K, np.zeros((1, K), dtype=np.float32))
    assert np.all(Y0 == 0) and np.all(A0 == 0)


@pytest.mark.parametrize("type_", [PN3T, PN4T])
def test_pn_gemv_closed_form_constant_codes(oracle, type_):
    """Every code n and every d equal: y = d * (n - z) * K * x for x = constant."""
    K, N = BLK[type_] * 4, 3
    z = {PN3T: 4, PN4T: 8}[type_]
    bits = {PN3T: 3, PN4T: 4}[type_]
    for n in range(2 * z):
        half = 0
        for j in range(5 if type_ == PN3T else 4):
            half |= n << (bits * j)
        word = half | (half << 16)
        block = np.frombuffer((0x3A00).to_bytes(2, "little") + word.to_bytes(4, "little") * 8, dtype=np.uint8)
        W = np.tile(block, N * (K // BLK[type_]))
        Y, _ = oracle.gemv(type_, W, N, K, np.full((1, K), 0.5, dtype=np.float32))
        assert np.all(Y == 0.75 * (n - z) * K * 0.5)  # 0x3A00 = 0.75


def test_nvfp4_gemv_vs_numpy(oracle):
    N, K, M = 30, 128, 2
    codes, scales, g = synth.nvfp4_random(N, K, seed=9)
    codes, scales = codes.numpy(), scales.numpy()
    X = synth.activations_bf16(M, K, seed=9)
    Y, A = oracle.gemv_nvfp4(codes, scales, g, N, K, X)
    G = grid()
    nib = np.stack([codes & 15, codes >> 4], axis=-1).reshape(N, K)
    Wd = np.vectorize(G.get)(nib).astype(np.float64) * np.repeat(torch_e4m3(scales), 16, axis=1) * np.float64(np.float32(g))
    Xd = torch.from_numpy(X.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.allclose(Y, Xd @ Wd.T, rtol=1e-12, atol=1e-15)
    assert np.allclose(A, np.abs(Xd) @ np.abs(Wd).T, rtol=1e-12, atol=1e-15)
