"""The prefill path (pnq_gemm: any M, PN on the tcgen05 tensor cores with tf32 splits) against the
oracle's fp64 GEMV over the exactly decoded weights, within the GEMV bound; slices smaller than N
(the caller's scratch), K tails that do not fill a 32-wide step, and the scratch-size error."""
import numpy as np
import pytest
import torch

import block_quantized_weight_pn3t_gb300 as pnq
from block_quantized_weight_pn3t_gb300 import synth
from gpu_util import assert_within_tolerance

pytestmark = pytest.mark.gpu

BLK = {pnq.PN3T: 80, pnq.PN4T: 64}


def run(type_, W, N, K, X, slice_rows=0):
    Xd = torch.from_numpy(X).cuda()
    Y = pnq.gemm(type_, W.cuda(), Xd, N, K, slice_rows=slice_rows)
    torch.cuda.synchronize()
    assert pnq.device_error() == 0
    return Y.cpu().numpy()


@pytest.mark.parametrize("type_", [pnq.PN3T, pnq.PN4T])
@pytest.mark.parametrize("M", [17, 64, 512])
@pytest.mark.parametrize("N,nblk", [(300, 16), (130, 40), (129, 3)])
def test_prefill_parity(oracle, type_, M, N, nblk):
    K = BLK[type_] * nblk
    seed = hash((type_, M, N, nblk)) % 1000
    W = synth.pn_random_blocks(type_, N, K, seed=seed)
    X = synth.activations(M, K, seed=seed + 1)
    Yr, Ar = oracle.gemv(type_, W.numpy(), N, K, X)
    Y = run(type_, W, N, K, X)
    assert_within_tolerance(Y, Yr, Ar, f"prefill type={type_} N={N} K={K} M={M}")


@pytest.mark.parametrize("type_", [pnq.PN3T, pnq.PN4T])
def test_prefill_slices(oracle, type_):
    """Scratch for 128-row slices: N = 300 runs as three slices, the last ragged."""
    N, K, M = 300, BLK[type_] * 8, 40
    W = synth.pn_random_blocks(type_, N, K, seed=5)
    X = synth.activations(M, K, seed=6)
    Yr, Ar = oracle.gemv(type_, W.numpy(), N, K, X)
    assert_within_tolerance(run(type_, W, N, K, X, slice_rows=128), Yr, Ar, f"prefill slices type={type_}")


def test_prefill_small_m_and_quantizer_weights(oracle):
    """M below 17 takes the same path; weights from the reference quantizer (zero rows, negative d)."""
    N, K = 256, 640
    w = synth.quantizer_weights(N, K, seed=8)
    W = torch.from_numpy(oracle.quantize(pnq.PN3T, w).reshape(-1))
    for M in (1, 5, 16):
        X = synth.activations(M, K, seed=M)
        Yr, Ar = oracle.gemv(pnq.PN3T, W.numpy(), N, K, X)
        assert_within_tolerance(run(pnq.PN3T, W, N, K, X), Yr, Ar, f"prefill quantizer M={M}")


def test_prefill_workload_sampled(oracle):
    """pn3t 17408 x 5120 at M = 512 (a 512-token prefill of the gate projection); sampled rows."""
    N, K, M = 17408, 5120, 512
    W = synth.pn_random_blocks(pnq.PN3T, N, K, seed=21, device="cuda")
    X = synth.activations(M, K, seed=22)
    Y = pnq.gemm(pnq.PN3T, W, torch.from_numpy(X).cuda(), N, K).cpu().numpy()
    rows = np.unique(np.concatenate([np.arange(3), np.arange(N - 3, N), np.random.default_rng(2).integers(0, N, 26)]))
    Wr = synth.pn_random_blocks(pnq.PN3T, N, K, seed=21, rows=torch.from_numpy(rows)).numpy()
    Yr, Ar = oracle.gemv(pnq.PN3T, Wr, len(rows), K, X)
    assert_within_tolerance(Y[:, rows], Yr, Ar, "prefill workload 17408x5120 M=512")
    assert pnq.device_error() == 0


def test_prefill_scratch_too_small():
    N, K, M = 256, 640, 32
    W = synth.pn_random_blocks(pnq.PN3T, N, K, seed=1).cuda()
    X = torch.zeros((M, K), dtype=torch.float32, device="cuda")
    need = pnq.gemm_scratch_bytes(pnq.PN3T, N, K, M, 128)
    assert need == 8 * K * (M + 128)
    with pytest.raises(pnq.PnqError) as e:
        pnq.gemm(pnq.PN3T, W, X, N, K, scratch=torch.empty((need - 16,), dtype=torch.uint8, device="cuda"))
    assert e.value.status == pnq.Status.ERR_SCRATCH
