"""pnq_gemv_noalloc: the GEMV entry point that allocates nothing (its cross-CTA partial sums use
the library's fixed 4 MiB device scratch). Kept in its own file, collected last, so the calls of
the other GPU tests run first. Results must equal pnq_gemv's bit for bit on two calls in a row
(the second call finds the scratch counters the first left zero), and a shape whose partial
sums do not fit must be refused before anything is launched."""
import numpy as np
import pytest
import torch

import block_quantized_weight_pn3t_gb300 as pnq
from block_quantized_weight_pn3t_gb300 import synth

pytestmark = pytest.mark.gpu

CASES = [(pnq.PN4T, 5120, 17408, 1), (pnq.PN4T, 5120, 6144, 4), (pnq.PN4T, 1024, 5120, 2),
         (pnq.PN3T, 17408, 5120, 1), (pnq.PN3T, 300, 1280, 3), (pnq.PN3T, 12288, 5120, 8)]


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


def test_noalloc_refuses_shapes_beyond_its_scratch():
    # 5120 x 17408 pn4t at M = 16: its partial sums (40 row tiles x 34 K units x 16 rows x 128)
    # need about 11 MB, more than the 4 MiB scratch
    N, K, M = 5120, 17408, 16
    W = synth.pn_random_blocks(pnq.PN4T, N, K, seed=3, device="cuda")
    X = torch.from_numpy(synth.activations(M, K, seed=4)).cuda()
    Y = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    rc = pnq.gemv_noalloc_ptr(pnq.PN4T, W.data_ptr(), N, K, X.data_ptr(), M, Y.data_ptr(), 0,
                              torch.cuda.current_stream().cuda_stream)
    assert rc == pnq.Status.ERR_SCRATCH
    torch.cuda.synchronize()
    assert bool((Y == 7.0).all())  # nothing was launched
    # the same call through pnq_gemv works (per-stream workspace)
    pnq.gemv(pnq.PN4T, W, X, N, K, Y=Y)
    torch.cuda.synchronize()
    assert pnq.device_error() == 0
