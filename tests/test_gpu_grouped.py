"""GPU grouped signed-integer formats (Q4G64/Q5G64/Q6G64/W8G32_F16S, "tensor-formats.md" sections 4
to 7) and the two GPU encoders, against the oracle:
  - dequantize: bit-exact; validate: equal flags;
  - GEMV: within |y - Y| <= 1e-5 * sum|w x| + 1e-6 of the oracle's fp64 sum;
  - the canonical encoder MAXABS_F16_RECIP_RNE_V1 on the GPU: planes bit-identical to the oracle's,
    rejected rows flagged;
  - the PN reference quantizer on the GPU: blocks bit-identical to the oracle's, rows with a
    non-finite weight flagged.
"""
import numpy as np
import pytest
import torch

import block_quantized_weight_pn3t_gb300 as pnq
from block_quantized_weight_pn3t_gb300 import synth
from gpu_util import assert_within_tolerance, device_bytes

pytestmark = pytest.mark.gpu

TYPES = [pnq.Q4G64_F16S, pnq.Q5G64_F16S, pnq.Q6G64_F16S, pnq.W8G32_F16S]


def random_planes(type_, N, K, seed):
    """Valid planes: random codes (W8 without 0x80), scales finite positive with a few +0 groups
    (their codes zeroed) and the smallest subnormal."""
    bits, G = pnq.GROUPED[type_]
    rng = np.random.default_rng(seed)
    slo, shi, ssc = pnq.grouped_plane_shapes(type_, N, K)
    lo = rng.integers(0, 256, size=slo, dtype=np.uint8)
    if bits == 8:
        lo[lo == 0x80] = 0x81
    hi = None if shi is None else rng.integers(0, 256, size=shi, dtype=np.uint8)
    sc = rng.integers(0x0001, 0x7C00, size=ssc, dtype=np.uint16)
    sc[:, 0] = 0x0001
    if N > 2 and ssc[1] > 1:  # a +0 group over zero codes
        sc[2, 1] = 0
        k0, k1 = G, min(2 * G, K)
        if bits == 8:
            lo[2, k0:k1] = 0
        else:
            lo[2, k0 // 2:k1 // 2] = 0
            if bits == 5:
                hi[2, k0 // 8:k1 // 8] = 0
            if bits == 6:
                hi[2, k0 // 4:k1 // 4] = 0
    return lo, hi, sc


def to_dev(lo, hi, sc):
    return (torch.from_numpy(lo).cuda(), None if hi is None else torch.from_numpy(hi).cuda(),
            torch.from_numpy(sc.view(np.int16)).cuda())


@pytest.mark.parametrize("type_", TYPES)
@pytest.mark.parametrize("N,K", [(1, 8), (37, 200), (130, 512), (9, 1032)])
def test_dequantize_bit_exact(oracle, type_, N, K):
    lo, hi, sc = random_planes(type_, N, K, seed=N + K)
    out = pnq.dequantize_row(type_, to_dev(lo, hi, sc), N, K).cpu().numpy()
    ref = oracle.dequantize_grouped(type_, lo, hi, sc, N, K)
    assert np.array_equal(out.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("type_", TYPES)
def test_validate(oracle, type_):
    bits, G = pnq.GROUPED[type_]
    N, K = 24, 3 * G + 16
    lo, hi, sc = random_planes(type_, N, K, seed=5)
    sc[4, 0] |= 0x8000
    sc[5, 1] = 0x7C00
    sc[6, 2] = 0x7D01
    sc[7, 0] = 0x0000  # +0 over random (almost surely nonzero) codes
    sc[8, 3] = 0x8000  # -0
    if bits == 8:
        lo[9, 17] = 0x80
    flags = pnq.validate_row(type_, to_dev(lo, hi, sc), N, K).cpu().numpy()
    ref = oracle.validate_grouped(type_, lo, hi, sc, N, K)
    assert np.array_equal(flags, ref)
    assert ref[4] and ref[5] and ref[6] and ref[7] and ref[8] and (ref[9] or bits != 8) and not ref[0]


@pytest.mark.parametrize("type_", TYPES)
@pytest.mark.parametrize("N,K", [(1, 64), (33, 520), (200, 2048)])
@pytest.mark.parametrize("M", [1, 3, 16])
def test_gemv(oracle, type_, N, K, M):
    w = synth.quantizer_weights(N, K, seed=N + K + M)
    lo, hi, sc = oracle.quantize_grouped(type_, w)
    X = synth.activations(M, K, seed=M)
    Y = pnq.gemv(type_, to_dev(lo, hi, sc), torch.from_numpy(X).cuda(), N, K).cpu().numpy()
    Yr, Ar = oracle.gemv_grouped(type_, lo, hi, sc, N, K, X)
    assert_within_tolerance(Y, Yr, Ar, f"type={type_} N={N} K={K} M={M}")


@pytest.mark.parametrize("type_", TYPES)
def test_gemv_workload_sampled(oracle, type_):
    """17408 x 5120 at M = 1 with planes encoded on the GPU; sampled rows checked on the host."""
    N, K = 17408, 5120
    w = torch.from_numpy(synth.quantizer_weights(N, K, seed=77)).cuda()
    planes, status = pnq.quantize_row(type_, w)
    assert int(status.sum()) == 0
    X = synth.activations(1, K, seed=78)
    Y = pnq.gemv(type_, planes, torch.from_numpy(X).cuda(), N, K).cpu().numpy()
    rows = np.unique(np.concatenate([np.arange(4), np.arange(N - 4, N), np.random.default_rng(1).integers(0, N, 48)]))
    lo, hi, sc = (None if t is None else t.cpu().numpy() for t in planes)
    sc = sc.view(np.uint16)
    Yr, Ar = oracle.gemv_grouped(type_, lo[rows], None if hi is None else hi[rows], sc[rows], len(rows), K, X)
    assert_within_tolerance(Y[:, rows], Yr, Ar, f"type={type_} workload")


def encoder_inputs(type_, seed):
    """Rows that exercise the encoder: normal weights with outliers, an all-zero row, tiny groups
    (the 2^-24 rescue), values near rounding ties of x * inv, a partial last group, and two
    rejected rows (an overflowing scale, a NaN)."""
    bits, G = pnq.GROUPED[type_]
    qmax = {4: 7, 5: 15, 6: 31, 8: 127}[bits]
    K = 4 * G + 8
    w = synth.quantizer_weights(40, K, seed=seed)
    rng = np.random.default_rng(seed)
    w[2, :G] = np.float32(2.0 ** -30)
    w[3, :] = (rng.integers(-qmax, qmax, size=K) + 0.5).astype(np.float32) * np.float32(0.25)
    w[3, ::G] = np.float32(qmax * 0.25)
    w[4, :] = np.nextafter(w[3, :], np.float32(np.inf))
    w[5, :] = np.nextafter(w[3, :], np.float32(-np.inf))
    w[6, 5] = np.float32(70000.0 * qmax)  # scale overflows binary16
    w[7, 9] = np.nan
    return w, {6, 7}


@pytest.mark.parametrize("type_", TYPES)
def test_encoder_bit_exact(oracle, type_):
    w, rejected = encoder_inputs(type_, seed=42)
    n, K = w.shape
    planes, status = pnq.quantize_row(type_, torch.from_numpy(w).cuda())
    status = status.cpu().numpy()
    assert set(np.nonzero(status)[0]) == rejected
    ok = np.array([r for r in range(n) if r not in rejected])
    lo, hi, sc = oracle.quantize_grouped(type_, w[ok])
    glo, ghi, gsc = (None if t is None else t.cpu().numpy() for t in planes)
    assert np.array_equal(glo[ok], lo)
    assert (hi is None and ghi is None) or np.array_equal(ghi[ok], hi)
    assert np.array_equal(gsc.view(np.uint16)[ok], sc)
    for r in rejected:
        with pytest.raises(ValueError):
            oracle.quantize_grouped(type_, w[r:r + 1])


@pytest.mark.parametrize("type_", TYPES)
def test_alignment_and_shape_errors(type_):
    bits, G = pnq.GROUPED[type_]
    N, K = 4, 64
    lo, hi, sc = to_dev(*random_planes(type_, N, K, seed=1))
    bad_lo, _keep = device_bytes(lo.cpu().numpy(), 2)
    with pytest.raises(pnq.PnqError) as e:
        pnq.dequantize_row(type_, (bad_lo, hi, sc), N, K)
    assert e.value.status == pnq.Status.ERR_ALIGN
    with pytest.raises(pnq.PnqError) as e:
        pnq.dequantize_row(type_, (lo, hi, sc), N, 60)
    assert e.value.status == pnq.Status.ERR_SHAPE


@pytest.mark.parametrize("type_", [pnq.PN3T, pnq.PN4T])
def test_pn_quantizer_bit_exact(oracle, type_):
    """The GPU reference quantizer chooses the oracle's d and codes for every block: normal
    weights with outliers, an all-zero row, an all-positive row (negative d), tiny blocks (fp16
    subnormal scales), huge blocks (candidates that overflow fp16 and are skipped)."""
    blk = pnq.BLOCK_WEIGHTS[type_]
    N, K = 48, blk * 24
    w = synth.quantizer_weights(N, K, seed=9)
    w[2] *= np.float32(1e-6)
    w[3] *= np.float32(3e-8)
    w[4] *= np.float32(2.0e6)
    w[5, :blk] = np.float32(0.5)  # constant block: several candidates tie on error
    w[6, :blk] = -np.float32(0.5)
    out, status = pnq.quantize_row(type_, torch.from_numpy(w).cuda())
    assert int(status.sum()) == 0
    ref = oracle.quantize(type_, w)
    got = out.cpu().numpy().reshape(N, -1)
    bad = np.nonzero((got != ref).any(axis=1))[0]
    assert bad.size == 0, f"rows {bad[:8]} differ"


@pytest.mark.parametrize("type_", [pnq.PN3T, pnq.PN4T])
def test_pn_quantizer_rejects_non_finite_rows(oracle, type_):
    blk = pnq.BLOCK_WEIGHTS[type_]
    N, K = 6, blk * 4
    w = synth.quantizer_weights(N, K, seed=10)
    w[1, 7] = np.inf
    w[4, blk + 3] = np.nan
    out, status = pnq.quantize_row(type_, torch.from_numpy(w).cuda())
    assert list(status.cpu().numpy()) == [0, 1, 0, 0, 1, 0]
    ok = [0, 2, 3, 5]
    assert np.array_equal(out.cpu().numpy().reshape(N, -1)[ok], oracle.quantize(type_, w[ok]))


def test_nvfp4_clip_search_bit_exact(oracle):
    """The GPU clip search keeps the oracle's multiplier, scales and codes in every group
    (TandemLLM "Quantisation and profiles", section "The clip search")."""
    N, K, g = 64, 512, 0.003
    w = synth.quantizer_weights(N, K, seed=31, sigma=0.05)
    w[2, :16] = 0.0
    w[3, :32] = -0.0
    w[4] *= np.float32(1e-4)  # tiny groups: scales near the E4M3 subnormals
    rng = np.random.default_rng(2)
    act = rng.uniform(0.0, 4.0, size=K).astype(np.float32)
    act[::7] = 0.0
    codes, scales, status = pnq.quantize_nvfp4_clip(torch.from_numpy(w).cuda(), torch.from_numpy(act).cuda(), g)
    assert int(status.sum()) == 0
    rc, rs, _ = oracle.quantize_nvfp4_clip(w, act, g)
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


def test_nvfp4_clip_search_rejects_rows_and_bad_scale(oracle):
    N, K = 4, 64
    w = synth.quantizer_weights(N, K, seed=32)
    w[2, 5] = np.inf
    act = np.ones(K, dtype=np.float32)
    codes, scales, status = pnq.quantize_nvfp4_clip(torch.from_numpy(w).cuda(), torch.from_numpy(act).cuda(), 0.01)
    assert list(status.cpu().numpy()) == [0, 0, 1, 0]
    with pytest.raises(pnq.PnqError) as e:
        pnq.quantize_nvfp4_clip(torch.from_numpy(w).cuda(), torch.from_numpy(act).cuda(), 0.0)
    assert e.value.status == pnq.Status.ERR_VALUE
