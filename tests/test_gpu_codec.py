"""GPU dequantize and validate against the oracle: bit-exact (NaN payloads compared by class)."""
import numpy as np
import pytest
import torch

import block_quantized_weight_pn3t_gb300 as pnq
from block_quantized_weight_pn3t_gb300 import synth
from gpu_util import device_bytes

pytestmark = pytest.mark.gpu

BLK = {pnq.PN3T: 80, pnq.PN4T: 64}


def same_bits_or_nan(a, b):
    a = np.asarray(a, dtype=np.float32)
    b = np.asarray(b, dtype=np.float32)
    nan = np.isnan(a) | np.isnan(b)
    return np.array_equal(np.isnan(a), np.isnan(b)) and np.array_equal(a.view(np.uint32)[~nan], b.view(np.uint32)[~nan])


@pytest.mark.parametrize("type_", [pnq.PN3T, pnq.PN4T])
@pytest.mark.parametrize("offset", [0, 2, 4, 6, 8, 14])
def test_pn_dequantize_bit_exact(oracle, type_, offset):
    N, K = 37, BLK[type_] * 24
    W = synth.pn_random_blocks(type_, N, K, seed=10 + offset).numpy()
    Wd, _ = device_bytes(W, offset)
    out = pnq.dequantize_row(type_, Wd, N, K)
    ref = oracle.dequantize(type_, W, N, K)
    assert same_bits_or_nan(out.cpu().numpy(), ref)


@pytest.mark.parametrize("type_", [pnq.PN3T, pnq.PN4T])
def test_pn_dequantize_quantizer_packed_and_signed_zero(oracle, type_):
    N, K = 256, BLK[type_] * 8
    W = oracle.quantize(type_, synth.quantizer_weights(N, K, seed=1))
    out = pnq.dequantize_row(type_, torch.from_numpy(W).cuda(), N, K).cpu().numpy()
    ref = oracle.dequantize(type_, W, N, K)
    assert np.array_equal(out.view(np.uint32), ref.view(np.uint32))
    assert np.any((ref == 0) & np.signbit(ref))  # -0.0 from code z with negative d is covered


@pytest.mark.parametrize("type_", [pnq.PN3T, pnq.PN4T])
def test_pn_dequantize_nonfinite_d(oracle, type_):
    N, K = 6, BLK[type_] * 2
    W = synth.pn_random_blocks(type_, N, K, seed=4).numpy().copy()
    for r, d in enumerate((0x7C00, 0xFC00, 0x7E00, 0x7C01, 0xFE00, 0x7BFF)):
        W[r, 34:36] = np.frombuffer(d.to_bytes(2, "little"), dtype=np.uint8)
    out = pnq.dequantize_row(type_, torch.from_numpy(W).cuda(), N, K).cpu().numpy()
    assert same_bits_or_nan(out, oracle.dequantize(type_, W, N, K))


def test_nvfp4_dequantize_every_code_and_scale(oracle):
    codes = np.zeros((256, 8), dtype=np.uint8)
    scales = np.arange(256, dtype=np.uint8).reshape(256, 1)
    codes[:] = [(2 * i) | ((2 * i + 1) << 4) for i in range(8)]
    for g in (1.0, 0.01, 3.0e-5, 7.5e30):
        out = pnq.dequantize_row(pnq.NVFP4, (torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda(), g), 256, 16)
        assert same_bits_or_nan(out.cpu().numpy(), oracle.dequantize_nvfp4(codes, scales, g, 256, 16))


@pytest.mark.parametrize("offset", [0, 1, 3])
def test_nvfp4_dequantize_random(oracle, offset):
    N, K = 50, 272
    codes, scales, g = synth.nvfp4_random(N, K, seed=6)
    cd, _ = device_bytes(codes.numpy(), offset)
    sd, _ = device_bytes(scales.numpy(), offset)
    out = pnq.dequantize_row(pnq.NVFP4, (cd, sd, g), N, K)
    assert same_bits_or_nan(out.cpu().numpy(), oracle.dequantize_nvfp4(codes.numpy(), scales.numpy(), g, N, K))


def test_nvfp4_div_dequantize_every_code_and_scale(oracle):
    codes = np.zeros((256, 8), dtype=np.uint8)
    scales = np.arange(256, dtype=np.uint8).reshape(256, 1)
    codes[:] = [(2 * i) | ((2 * i + 1) << 4) for i in range(8)]
    for dw in (1.0, 0.37, 3.0e-5, 7.5e30, 1.0e-40):
        out = pnq.dequantize_row(pnq.NVFP4_DIV, (torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda(), dw),
                                 256, 16)
        assert same_bits_or_nan(out.cpu().numpy(), oracle.dequantize_nvfp4_div(codes, scales, dw, 256, 16))


@pytest.mark.parametrize("offset", [0, 1, 3])
def test_nvfp4_div_dequantize_random(oracle, offset):
    N, K = 50, 272
    codes, scales, _ = synth.nvfp4_random(N, K, seed=7)
    cd, _ = device_bytes(codes.numpy(), offset)
    sd, _ = device_bytes(scales.numpy(), offset)
    out = pnq.dequantize_row(pnq.NVFP4_DIV, (cd, sd, 0.37), N, K)
    assert same_bits_or_nan(out.cpu().numpy(), oracle.dequantize_nvfp4_div(codes.numpy(), scales.numpy(), 0.37, N, K))


def test_validate_nvfp4_div(oracle):
    """Same validity rule as the multiplier reading: the divisor must be finite and > 0."""
    N, K = 40, 64
    codes, scales, _ = synth.nvfp4_random(N, K, seed=8)
    s = scales.numpy().copy()
    s[3, 1] = 0x80
    s[7, 0] = 0x7F
    for dw in (0.37, 1.0e-45, 0.0, -1.0, float("inf"), float("nan")):
        flags = pnq.validate_row(pnq.NVFP4_DIV, (codes.cuda(), torch.from_numpy(s).cuda(), dw), N, K).cpu().numpy()
        assert np.array_equal(flags, oracle.validate_nvfp4(s, dw, N, K))


def inject_bad_rows(type_, W, K, rng):
    """Rows with non-finite d (0x7C00, 0xFC00, 0x7E00, 0x7C01) and, for pn3t, set reserved bits."""
    nb = K // BLK[type_]
    W = W.copy()
    rows = rng.choice(W.shape[0], 12, replace=False)
    for i, r in enumerate(rows[:8]):
        b = rng.integers(nb)
        d = (0x7C00, 0xFC00, 0x7E00, 0x7C01)[i % 4]
        W[r, 34 * b: 34 * b + 2] = np.frombuffer(d.to_bytes(2, "little"), dtype=np.uint8)
    for r in rows[8:]:
        b, word = rng.integers(nb), rng.integers(8)
        o = 34 * b + 2 + 4 * word
        v = int.from_bytes(bytes(W[r, o: o + 4]), "little") | (1 << int(rng.choice([15, 31])))
        W[r, o: o + 4] = np.frombuffer(v.to_bytes(4, "little"), dtype=np.uint8)
    return W


@pytest.mark.parametrize("type_", [pnq.PN3T, pnq.PN4T])
def test_validate_down_projection_size(oracle, type_):
    """5120 rows x 17408 (pn4t down-projection shape; pn3t at 17440 = 218 blocks)."""
    rng = np.random.default_rng(0)
    N, K = 5120, (17408 if type_ == pnq.PN4T else 17440)
    W = inject_bad_rows(type_, synth.pn_random_blocks(type_, N, K, seed=12).numpy(), K, rng)
    flags = pnq.validate_row(type_, torch.from_numpy(W).cuda(), N, K).cpu().numpy()
    ref = oracle.validate(type_, W, N, K)
    assert np.array_equal(flags, ref)
    assert ref.sum() == (12 if type_ == pnq.PN3T else 8)


@pytest.mark.parametrize("offset", [0, 2, 6])
def test_validate_unaligned(oracle, offset):
    rng = np.random.default_rng(1)
    N, K = 300, 80 * 5
    W = inject_bad_rows(pnq.PN3T, synth.pn_random_blocks(pnq.PN3T, N, K, seed=2).numpy(), K, rng)
    Wd, _ = device_bytes(W, offset)
    assert np.array_equal(pnq.validate_row(pnq.PN3T, Wd, N, K).cpu().numpy(), oracle.validate(pnq.PN3T, W, N, K))


def test_validate_nvfp4(oracle):
    N, K = 1000, 512
    codes, scales, g = synth.nvfp4_random(N, K, seed=5)
    s = scales.numpy().copy()
    rng = np.random.default_rng(2)
    for r, bad in zip(rng.choice(N, 8, replace=False), (0x80, 0xB8, 0x7F, 0xFF, 0x80, 0xC0, 0x7F, 0xFE)):
        s[r, rng.integers(K // 16)] = bad
    c = codes.cuda()
    for gv in (g, 0.0, -1.0, float("inf"), float("nan")):
        flags = pnq.validate_row(pnq.NVFP4, (c, torch.from_numpy(s).cuda(), gv), N, K).cpu().numpy()
        assert np.array_equal(flags, oracle.validate_nvfp4(s, gv, N, K))
