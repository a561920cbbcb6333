"""GPU GEMV against the fp64 oracle: |y - y_ref| <= 1e-5 * sum|w x| + 1e-6 per element.

Covers both paths (tensor-core fast path for aligned weights with (K/BLK) % 8 == 0 or
NVFP4 K % 256 == 0; generic path otherwise), every M from the matrix-vector (1..4) and
small-batch (5..16) ranges, ragged N, alignment offsets, the workload sizes (sampled rows),
exact closed forms, canaries past the output, determinism, and forced tile / grid / stage
configurations.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import block_quantized_weight_pn3t_gb300 as pnq
from block_quantized_weight_pn3t_gb300 import synth
from gpu_util import assert_within_tolerance, canary_intact, device_bytes, f32_with_canary

pytestmark = pytest.mark.gpu

BLK = {pnq.PN3T: 80, pnq.PN4T: 64}
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_pn(type_, W_np, N, K, X_np, offset=0):
    Wd, _back = device_bytes(W_np, offset)
    M = X_np.shape[0]
    buf, Y = f32_with_canary(M, N)
    pnq.gemv(type_, Wd, torch.from_numpy(X_np).cuda(), N, K, Y=Y)
    torch.cuda.synchronize()
    assert canary_intact(buf, M * N)
    return Y.cpu().numpy()


def run_nv(codes, scales, g, N, K, Xb, offset=0):
    cd, _b1 = device_bytes(codes, offset)
    sd, _b2 = device_bytes(scales, offset)
    M = Xb.shape[0]
    buf, Y = f32_with_canary(M, N)
    pnq.gemv(pnq.NVFP4, (cd, sd, g), torch.from_numpy(Xb.view(np.int16)).cuda(), N, K, Y=Y)
    torch.cuda.synchronize()
    assert canary_intact(buf, M * N)
    return Y.cpu().numpy()


def test_config1_quantizer_packed(oracle):
    """pn3t N=256, K=640, weights N(0, 0.02) with outliers, packed by the reference
    quantizer, zero row and negative-d row; M = 1 (and 2, 4)."""
    N, K = 256, 640
    W = oracle.quantize(pnq.PN3T, synth.quantizer_weights(N, K, seed=1))
    for M in (1, 2, 4):
        X = synth.activations(M, K, seed=M)
        Y = run_pn(pnq.PN3T, W, N, K, X)
        Yr, Ar = oracle.gemv(pnq.PN3T, W, N, K, X)
        assert_within_tolerance(Y, Yr, Ar, f"config1 M={M}")
        assert np.all(Y[:, 0] == 0)  # canonical zero row


@pytest.mark.parametrize("type_", [pnq.PN3T, pnq.PN4T])
@pytest.mark.parametrize("nblk", [8, 24, 40, 3])
@pytest.mark.parametrize("N", [1, 33, 130])
@pytest.mark.parametrize("M", [1, 2, 4, 5, 7, 8, 16])
def test_pn_shapes(oracle, type_, nblk, N, M):
    K = BLK[type_] * nblk
    seed = hash((type_, nblk, N, M)) % 1000
    W = synth.pn_random_blocks(type_, N, K, seed=seed).numpy()
    X = synth.activations(M, K, seed=seed)
    Yr, Ar = oracle.gemv(type_, W, N, K, X)
    for offset in (0, 6):  # 6: 2-byte aligned only -> generic path
        Y = run_pn(type_, W, N, K, X, offset)
        assert_within_tolerance(Y, Yr, Ar, f"type={type_} K={K} N={N} M={M} off={offset}")


@pytest.mark.parametrize("K", [256, 768, 80, 528])
@pytest.mark.parametrize("N", [1, 33, 130])
@pytest.mark.parametrize("M", [1, 3, 4, 5, 8, 9, 16])
def test_nvfp4_shapes(oracle, K, N, M):
    seed = hash((K, N, M)) % 1000
    codes, scales, g = synth.nvfp4_random(N, K, seed=seed)
    codes, scales = codes.numpy(), scales.numpy()
    Xb = synth.activations_bf16(M, K, seed=seed)
    Yr, Ar = oracle.gemv_nvfp4(codes, scales, g, N, K, Xb)
    for offset in (0, 1):  # 1: unaligned codes/scales -> generic path
        Y = run_nv(codes, scales, g, N, K, Xb, offset)
        assert_within_tolerance(Y, Yr, Ar, f"nvfp4 K={K} N={N} M={M} off={offset}")


def run_nv_div(codes, scales, dw, N, K, Xb, offset=0):
    cd, _b1 = device_bytes(codes, offset)
    sd, _b2 = device_bytes(scales, offset)
    M = Xb.shape[0]
    buf, Y = f32_with_canary(M, N)
    pnq.gemv(pnq.NVFP4_DIV, (cd, sd, dw), torch.from_numpy(Xb.view(np.int16)).cuda(), N, K, Y=Y)
    torch.cuda.synchronize()
    assert canary_intact(buf, M * N)
    return Y.cpu().numpy()


@pytest.mark.parametrize("K", [256, 768, 528])
@pytest.mark.parametrize("N", [1, 33, 130])
@pytest.mark.parametrize("M", [1, 4, 16])
@pytest.mark.parametrize("dw", [0.37, 2.0e38])
def test_nvfp4_div_shapes(oracle, K, N, M, dw):
    """NVFP4 with the global field as a divisor d_w ("tensor-formats.md" section 3.3). d_w = 2e38:
    1 / d_w is not a normal fp32 number, so every path divides each output by d_w (x is scaled
    by 2^100 to keep the products away from the bound's absolute term)."""
    seed = hash((K, N, M, dw)) % 1000
    codes, scales, _ = synth.nvfp4_random(N, K, seed=seed)
    codes, scales = codes.numpy(), scales.numpy()
    Xb = synth.activations_bf16(M, K, seed=seed)
    if dw > 1e30:
        Xb = (Xb.astype(np.uint32) + (100 << 7)).astype(np.uint16)  # x * 2^100 (exponent field + 100)
    Yr, Ar = oracle.gemv_nvfp4_div(codes, scales, dw, N, K, Xb)
    for offset in (0, 1):  # 1: unaligned codes/scales -> generic path
        Y = run_nv_div(codes, scales, dw, N, K, Xb, offset)
        assert_within_tolerance(Y, Yr, Ar, f"nvfp4/dw K={K} N={N} M={M} dw={dw} off={offset}")


@pytest.mark.parametrize("N,K", [(17408, 5120), (5120, 17408)])
@pytest.mark.parametrize("M", [1, 4])
def test_nvfp4_div_workload_sampled(oracle, N, K, M):
    codes, scales, _ = synth.nvfp4_random(N, K, seed=79, device="cuda")
    dw = 0.0123
    Xb = synth.activations_bf16(M, K, seed=80)
    Y = pnq.gemv(pnq.NVFP4_DIV, (codes, scales, dw), torch.from_numpy(Xb.view(np.int16)).cuda(), N, K).cpu().numpy()
    rows = sampled_rows(N)
    cr, sr, _ = synth.nvfp4_random(N, K, seed=79, rows=torch.from_numpy(rows))
    Yr, Ar = oracle.gemv_nvfp4_div(cr.numpy(), sr.numpy(), dw, len(rows), K, Xb)
    assert_within_tolerance(Y[:, rows], Yr, Ar, f"nvfp4/dw {N}x{K} M={M}")


@pytest.mark.parametrize("type_", [pnq.PN3T, pnq.PN4T])
@pytest.mark.parametrize("offset", [0, 2])
def test_one_hot_x_gives_exact_column(oracle, type_, offset):
    """x = e_k: y is the dequantized column k bit for bit (one nonzero product, exact scaling)."""
    N, K = 70, BLK[type_] * 16
    W = synth.pn_random_blocks(type_, N, K, seed=3).numpy()
    Wd = oracle.dequantize(type_, W, N, K)
    ks = [0, 1, BLK[type_] - 1, BLK[type_], 5 * BLK[type_] + 7, K - 1]
    X = np.zeros((len(ks), K), dtype=np.float32)
    for i, k in enumerate(ks):
        X[i, k] = 1.0
    Y = run_pn(type_, W, N, K, X, offset)
    for i, k in enumerate(ks):
        assert np.array_equal(Y[i], Wd[:, k]), (type_, k)


def test_zero_x_and_extreme_magnitudes(oracle):
    N, K = 64, 80 * 16
    W = synth.pn_random_blocks(pnq.PN3T, N, K, seed=9).numpy()
    Y = run_pn(pnq.PN3T, W, N, K, np.zeros((2, K), dtype=np.float32))
    assert np.all(Y == 0)
    base = synth.activations(3, K, seed=9)
    for scale in (1e30, 1e10, 1e-10, 1e-30):
        X = (base * np.float32(scale)).astype(np.float32)
        Yr, Ar = oracle.gemv(pnq.PN3T, W, N, K, X)
        for offset in (0, 2):
            assert_within_tolerance(run_pn(pnq.PN3T, W, N, K, X, offset), Yr, Ar, f"scale={scale} off={offset}")
    # a row of x spanning many binades (fp16 range is per slice of K, not per element)
    X = base.copy()
    X[0, ::7] *= np.float32(1e8)
    X[1, ::5] *= np.float32(1e-8)
    Yr, Ar = oracle.gemv(pnq.PN3T, W, N, K, X)
    assert_within_tolerance(run_pn(pnq.PN3T, W, N, K, X), Yr, Ar, "wide dynamic range")


def test_deterministic():
    N, K, M = 4096, 64 * 272, 4
    W = synth.pn_random_blocks(pnq.PN4T, N, K, seed=5, device="cuda")
    X = torch.from_numpy(synth.activations(M, K, seed=5)).cuda()
    a = pnq.gemv(pnq.PN4T, W, X, N, K).cpu().numpy()
    b = pnq.gemv(pnq.PN4T, W, X, N, K).cpu().numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def sampled_rows(N, n=48, seed=0):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, 1, 15, 16, 63, 64, N - 1], rng.choice(N, n, replace=False)]))


@pytest.mark.parametrize("type_,N,U,M", [(pnq.PN4T, 777, 34, 1), (pnq.PN3T, 300, 17, 1), (pnq.PN4T, 40, 33, 1),
                                         (pnq.PN3T, 2000, 25, 1), (pnq.PN4T, 161, 20, 2), (pnq.PN3T, 999, 12, 3),
                                         (pnq.PN4T, 153, 16, 4), (pnq.PN4T, 1500, 34, 6), (pnq.PN3T, 700, 12, 7),
                                         (pnq.PN4T, 4000, 20, 5), (pnq.PN3T, 2900, 9, 8), (pnq.PN4T, 5000, 34, 2)])
def test_pn_row_segments(oracle, type_, N, U, M):
    """Rows long enough to be cut into K segments (U = K units of 8 blocks), with segments of unequal
    length and CTAs whose last 16-row group is ragged; at M = 5..8 two n8 tiles per task; rows
    whose plan splits K over a cluster (unequal unit counts per CTA)."""
    K = BLK[type_] * 8 * U
    seed = 31 * U + N
    W = synth.pn_random_blocks(type_, N, K, seed=seed).numpy()
    X = synth.activations(M, K, seed=seed)
    Yr, Ar = oracle.gemv(type_, W, N, K, X)
    assert_within_tolerance(run_pn(type_, W, N, K, X), Yr, Ar, f"type={type_} N={N} U={U} M={M}")


def d_extremes(type_, N, seed):
    """PN blocks whose d runs over every fp16 exponent field 0..30 with both signs (so subnormals,
    the smallest and largest normals and 65504 = 0x7BFF appear), +0 and -0 over codes that are not
    z, and random fractions; codes random."""
    K_blocks = 8 * 4
    W = synth.pn_random_blocks(type_, N, BLK[type_] * K_blocks, seed=seed).numpy().reshape(N, K_blocks, 34).copy()
    rng = np.random.default_rng(seed)
    d = np.empty((N, K_blocks), dtype=np.uint16)
    vals = [(s << 15) | (e << 10) | f for e in range(31) for s in (0, 1) for f in (0, 1, 0x3FF, 0x155)]
    vals += [0x0000, 0x8000, 0x0001, 0x8001, 0x03FF, 0x7BFF, 0xFBFF, 0x0400]
    flat = d.reshape(-1)
    for i in range(flat.size):
        flat[i] = vals[i % len(vals)] if i < 3 * len(vals) else vals[rng.integers(len(vals))]
    W[:, :, 0] = d & 0xFF
    W[:, :, 1] = d >> 8
    if type_ == pnq.PN3T:  # keep the reserved bits clear
        W[:, :, 3] &= 0x7F
        W[:, :, 5] &= 0x7F
        for w in range(8):
            W[:, :, 2 + 4 * w + 1] &= 0x7F
            W[:, :, 2 + 4 * w + 3] &= 0x7F
    return W.reshape(N, -1), BLK[type_] * K_blocks


@pytest.mark.parametrize("type_", [pnq.PN3T, pnq.PN4T])
@pytest.mark.parametrize("M", [1, 4, 16])
def test_d_extremes(oracle, type_, M):
    """d over the whole fp16 range ("PN weight format", section Value: w = d * (n - z) is exact in
    fp32, a zero d gives a signed zero), on the fast path (aligned) and the generic path."""
    N = 160
    W, K = d_extremes(type_, N, seed=M)
    X = synth.activations(M, K, seed=M + 10)
    Yr, Ar = oracle.gemv(type_, W, N, K, X)
    assert np.all(np.isfinite(Yr))
    for offset in (0, 6):
        Y = run_pn(type_, W, N, K, X, offset)
        assert_within_tolerance(Y, Yr, Ar, f"d extremes type={type_} M={M} off={offset}")


LAYER = [("gate", pnq.PN3T, 17408, 5120), ("up", pnq.PN3T, 17408, 5120), ("q", pnq.PN3T, 12288, 5120),
         ("k", pnq.PN4T, 1024, 5120), ("v", pnq.PN4T, 1024, 5120), ("o", pnq.PN4T, 5120, 6144),
         ("down", pnq.PN4T, 5120, 17408)]


@pytest.mark.parametrize("name,type_,N,K", LAYER)
@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
def test_workload_shapes_sampled(oracle, name, type_, N, K, M):
    """One Qwen-27B-shaped layer's projections at full size (generated on the device from the
    seed); rows sampled and regenerated on the host for the oracle."""
    seed = 1000 + [l[0] for l in LAYER].index(name)
    W = synth.pn_random_blocks(type_, N, K, seed=seed, device="cuda")
    X = synth.activations(M, K, seed=seed + M)
    Y = pnq.gemv(type_, W, torch.from_numpy(X).cuda(), N, K).cpu().numpy()
    rows = sampled_rows(N)
    Wr = synth.pn_random_blocks(type_, N, K, seed=seed, rows=torch.from_numpy(rows)).numpy()
    assert np.array_equal(Wr, W[torch.from_numpy(rows).cuda()].cpu().numpy())  # host and device agree
    Yr, Ar = oracle.gemv(type_, Wr, len(rows), K, X)
    assert_within_tolerance(Y[:, rows], Yr, Ar, f"{name} M={M}")


@pytest.mark.parametrize("N,K", [(17408, 5120), (5120, 17408)])
@pytest.mark.parametrize("M", [1, 4, 8, 16])
def test_nvfp4_workload_sampled(oracle, N, K, M):
    codes, scales, g = synth.nvfp4_random(N, K, seed=77, device="cuda")
    Xb = synth.activations_bf16(M, K, seed=78)
    Y = pnq.gemv(pnq.NVFP4, (codes, scales, g), torch.from_numpy(Xb.view(np.int16)).cuda(), N, K).cpu().numpy()
    rows = sampled_rows(N)
    cr, sr, _ = synth.nvfp4_random(N, K, seed=77, rows=torch.from_numpy(rows))
    Yr, Ar = oracle.gemv_nvfp4(cr.numpy(), sr.numpy(), g, len(rows), K, Xb)
    assert_within_tolerance(Y[:, rows], Yr, Ar, f"nvfp4 {N}x{K} M={M}")


CHILD = r"""
import json, sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {root!r} + '/tests')
import numpy as np, torch
import block_quantized_weight_pn3t_gb300 as pnq
from block_quantized_weight_pn3t_gb300 import synth
import oracle
from gpu_util import assert_within_tolerance
out = []
for type_, N, K, M in [(124, 200, 80*48, 1), (125, 130, 64*80, 3), (125, 64, 64*8, 16), (124, 17, 80*16, 8),
                      (124, 1000, 80*16, 4), (125, 777, 64*272, 2), (124, 9, 80*8, 1), (125, 2500, 64*24, 12),
                      (125, 300, 64*272, 1), (124, 500, 80*136, 1)]:
    W = synth.pn_random_blocks(type_, N, K, seed=N + K)
    X = synth.activations(M, K, seed=M)
    for flags in (0, pnq.GEMV_STATIC_WEIGHTS):
        Y = pnq.gemv(type_, W.cuda(), torch.from_numpy(X).cuda(), N, K, flags=flags).cpu().numpy()
        Yr, Ar = oracle.gemv(type_, W.numpy(), N, K, X)
        assert_within_tolerance(Y, Yr, Ar, str((type_, N, K, M, flags)))
for N, K, M in [(130, 256*6, 1), (33, 256*9, 5), (64, 256*2, 16), (300, 256*10, 12), (777, 256*68, 2),
                (151, 256*21, 4)]:
    c, s, g = synth.nvfp4_random(N, K, seed=K)
    Xb = synth.activations_bf16(M, K, seed=K)
    Y = pnq.gemv(1004, (c.cuda(), s.cuda(), g), torch.from_numpy(Xb.view(np.int16)).cuda(), N, K).cpu().numpy()
    Yr, Ar = oracle.gemv_nvfp4(c.numpy(), s.numpy(), g, N, K, Xb)
    assert_within_tolerance(Y, Yr, Ar, str((N, K, M)))
torch.cuda.synchronize()
print(json.dumps({{"ok": True, "device_error": pnq.device_error()}}))
"""


@pytest.mark.parametrize("pn_cfg,nv_cfg", [("1,0,0,2", "2,0"), ("2,0,0,2", "1,0"), ("1,3,0,2", "1,6"),
                                            ("2,3,2,2", "2,3,2"), ("0,0,0,1", "2,4"), ("0,2,0,1", "1,3,1"),
                                            ("0,3,0,1", "0,5,2"), ("0,8,0,1", "0,3"), ("0,3,0,0", "1,4"),
                                            ("0,6,1,2", "2,6,1"), ("0,0,0,1,1", "0,0"), ("0,2,0,1,1", "0,0"),
                                            ("0,0,0,1,0,0,0,2", "0,0"), ("0,3,0,1,0,0,0,4", "0,0"),
                                            ("0,0,0,1,0,8,1,8", "0,0"), ("0,0,0,1,1,0,0,2", "0,0"),
                                            ("0,0,0,1", "0,0,0,2"), ("0,0,0,1", "0,0,0,4"), ("0,0,0,1", "0,0,0,8")])
def test_tile_and_grid_configs(pn_cfg, nv_cfg):
    """Forced configurations, read once per process (so each runs in a child): the PN path through
    PNQ_PN_CFG = "CTAs per cluster, weight stages, CTAs per SM, path, decode, x ahead, x apart, row
    clusters" (path 1 = the row stream, 2 = K-unit strips over clusters; decode 1 = the CUDA-core
    FMA decode of the row path, which shapes outside its plan leave to the generic path; x ahead =
    weight stages issued before x is requested; x apart 1 = x outside the weight ring; row clusters
    = CTAs splitting K in the row stream) and the NVFP4 path through PNQ_NV_CFG = "CTAs per
    cluster, weight stages, CTAs per SM, row clusters" (0 = automatic)."""
    env = dict(os.environ, PNQ_PN_CFG=pn_cfg, PNQ_NV_CFG=nv_cfg, PNQ_FORCE_KERNEL="mma")
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT)], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res == {"ok": True, "device_error": 0}


def test_no_device_error_recorded():
    torch.cuda.synchronize()
    assert pnq.device_error() == 0
