"""pnq_gemv_noalloc: the GEMV entry point that allocates nothing. Kept in its own file, collected
last, so the calls of the other GPU tests run first. Results must equal pnq_gemv_ex's bit for bit
on two calls in a row, for PN and NVFP4 shapes, including the widest batch (M = 16) at the
down-projection size."""
import numpy as np
import pytest
import torch

import block_quantized_weight_pn3t_gb300 as pnq
from block_quantized_weight_pn3t_gb300 import synth

pytestmark = pytest.mark.gpu

CASES = [(pnq.PN4T, 5120, 17408, 1), (pnq.PN4T, 5120, 6144, 4), (pnq.PN4T, 1024, 5120, 2),
         (pnq.PN3T, 17408, 5120, 1), (pnq.PN3T, 300, 1280, 3), (pnq.PN3T, 12288, 5120, 8),
         (pnq.PN4T, 5120, 17408, 16)]
NV_CASES = [(17408, 5120, 1), (5120, 17408, 4), (5120, 17408, 8), (300, 2560, 3), (5120, 17408, 16)]


@pytest.mark.parametrize("type_,N,K,M", CASES)
def test_noalloc_matches_gemv_on_two_calls(type_, N, K, M):
    W = synth.pn_random_blocks(type_, N, K, seed=N + M, device="cuda")
    X = torch.from_numpy(synth.activations(M, K, seed=M)).cuda()
    ref = pnq.gemv(type_, W, X, N, K)
    first = pnq.gemv_noalloc(type_, W, X, N, K)
    second = pnq.gemv_noalloc(type_, W, X, N, K)
    torch.cuda.synchronize()
    r = ref.cpu().numpy().view(np.uint32)
    assert np.array_equal(first.cpu().numpy().view(np.uint32), r)
    assert np.array_equal(second.cpu().numpy().view(np.uint32), r)
    assert pnq.device_error() == 0


@pytest.mark.parametrize("N,K,M", NV_CASES)
def test_noalloc_nvfp4_matches_gemv_on_two_calls(N, K, M):
    codes, scales, g = synth.nvfp4_random(N, K, seed=N + M, device="cuda")
    X = torch.from_numpy(synth.activations_bf16(M, K, seed=M).view(np.int16)).cuda()
    ref = pnq.gemv(pnq.NVFP4, (codes, scales, g), X, N, K)
    first = pnq.gemv_noalloc(pnq.NVFP4, (codes, scales, g), X, N, K)
    second = pnq.gemv_noalloc(pnq.NVFP4, (codes, scales, g), X, N, K)
    torch.cuda.synchronize()
    r = ref.cpu().numpy().view(np.uint32)
    assert np.array_equal(first.cpu().numpy().view(np.uint32), r)
    assert np.array_equal(second.cpu().numpy().view(np.uint32), r)
    assert pnq.device_error() == 0
