"""The failure path of the bounded waits, on the GPU without faulting it: a wait that nothing
completes runs out after a short limit, the kernel records its site code in the device error word
and returns; pnq_device_error reports and clears the code; the context stays usable (a GEMV and a
no-alloc GEMV afterwards agree bit for bit and match the oracle)."""
import numpy as np
import pytest
import torch

import block_quantized_weight_pn3t_gb300 as pnq
from block_quantized_weight_pn3t_gb300 import synth
from gpu_util import assert_within_tolerance

pytestmark = pytest.mark.gpu

SELFTEST_SITE = 6


def test_wait_that_runs_out_is_reported_and_cleared(oracle):
    torch.cuda.synchronize()
    assert pnq.device_error() == 0
    pnq.selftest_wait(2000)  # 2 ms
    torch.cuda.synchronize()
    assert pnq.device_error() == SELFTEST_SITE
    assert pnq.device_error() == 0  # read-and-clear
    # the first code stays: two self-tests in a row report one code
    pnq.selftest_wait(500)
    pnq.selftest_wait(500)
    assert pnq.device_error() == SELFTEST_SITE
    assert pnq.device_error() == 0
    # the context is still usable: fast-path GEMVs run and agree
    N, K, M = 300, 80 * 64, 1
    W = synth.pn_random_blocks(pnq.PN3T, N, K, seed=3)
    X = synth.activations(M, K, seed=3)
    Wd, Xd = W.cuda(), torch.from_numpy(X).cuda()
    Y1 = pnq.gemv(pnq.PN3T, Wd, Xd, N, K).cpu().numpy()
    Y2 = pnq.gemv_noalloc(pnq.PN3T, Wd, Xd, N, K).cpu().numpy()
    assert np.array_equal(Y1.view(np.uint32), Y2.view(np.uint32))
    Yr, Ar = oracle.gemv(pnq.PN3T, W.numpy(), N, K, X)
    assert_within_tolerance(Y1, Yr, Ar, "after the self-test")
    assert pnq.device_error() == 0


def test_selftest_limit_is_checked():
    for bad in (0, 2000001):
        with pytest.raises(pnq.PnqError) as e:
            pnq.selftest_wait(bad)
        assert e.value.status == pnq.Status.ERR_VALUE
