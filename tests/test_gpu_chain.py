"""Dependent GEMV chains in the launch configuration the decode-step benchmark times.

Every GEMV runs with the static-weights flag (programmatic dependent launch: a launch may start
streaming its weights while the previous grid still runs), back to back on one side stream,
first eagerly and then captured in a CUDA graph and replayed. Unlike the benchmark, each GEMV's
activations here are the previous GEMV's output, and every output buffer is filled with NaN
before each run: a GEMV that read its x, or wrote its Y, before the previous grid had completed
would leave NaNs or stale values behind. Each stage is checked against the fp64 oracle on the
input it actually received, within |y - y_ref| <= 1e-5 * sum|w x| + 1e-6, and graph replays
must reproduce the eager run bit for bit.

The chain mixes the paths a decode step meets: pn3t and pn4t fast paths (one CTA per row tile
and stream-K grids), an NVFP4 stage fed through a bf16 conversion kernel (a dependency on an
ordinary kernel), and a last pn4t stage whose K (1920 = 30 blocks) takes the generic path with
a ragged N.
"""
import numpy as np
import pytest
import torch

import block_quantized_weight_pn3t_gb300 as pnq
from block_quantized_weight_pn3t_gb300 import synth
from gpu_util import assert_within_tolerance

pytestmark = pytest.mark.gpu

# (type, N, K): K of each stage is N of the stage before; x0 has K = 2560
CHAIN = [(pnq.PN3T, 5120, 2560), (pnq.PN4T, 2560, 5120), (pnq.NVFP4, 3200, 2560), (pnq.PN3T, 1920, 3200),
         (pnq.PN4T, 1000, 1920)]


def make_chain(M):
    stages = []
    for i, (t, N, K) in enumerate(CHAIN):
        if t == pnq.NVFP4:
            codes, scales, g = synth.nvfp4_random(N, K, seed=300 + i, device="cuda")
            xin = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")  # bf16 copy of the previous output
            stages.append({"t": t, "N": N, "K": K, "W": (codes, scales, g), "xin": xin})
        else:
            W = synth.pn_random_blocks(t, N, K, seed=300 + i, device="cuda")
            stages.append({"t": t, "N": N, "K": K, "W": W, "xin": None})
        stages[-1]["Y"] = torch.empty((M, N), dtype=torch.float32, device="cuda")
    x0 = torch.from_numpy(synth.activations(M, CHAIN[0][2], seed=301)).cuda()
    return x0, stages


def launch_chain(x0, stages):
    """The chain on the current stream: every GEMV with the static-weights flag."""
    x = x0
    for s in stages:
        if s["xin"] is not None:
            s["xin"].copy_(x)  # fp32 -> bf16 on the device (round to nearest even)
            x = s["xin"]
        pnq.gemv(s["t"], s["W"], x.view(torch.int16) if s["t"] == pnq.NVFP4 else x, s["N"], s["K"], Y=s["Y"],
                 flags=pnq.GEMV_STATIC_WEIGHTS)
        x = s["Y"]


def poison(stages):
    for s in stages:
        s["Y"].fill_(float("nan"))
        if s["xin"] is not None:
            s["xin"].fill_(float("nan"))


def check_against_oracle(oracle, x0, stages, M):
    x_host = x0.cpu().numpy()
    for i, s in enumerate(stages):
        Y = s["Y"].cpu().numpy()
        assert not np.isnan(Y).any(), f"stage {i}: NaN left in the output (a read or write ran early)"
        if s["t"] == pnq.NVFP4:
            codes, scales, g = s["W"]
            xb = s["xin"].view(torch.int16).cpu().numpy().view(np.uint16)
            Yr, Ar = oracle.gemv_nvfp4(codes.cpu().numpy(), scales.cpu().numpy(), g, s["N"], s["K"], xb)
        else:
            Yr, Ar = oracle.gemv(s["t"], s["W"].cpu().numpy(), s["N"], s["K"], x_host)
        assert_within_tolerance(Y, Yr, Ar, f"chain stage {i} {CHAIN[i]} M={M}")
        x_host = Y


@pytest.mark.parametrize("M", [1, 4, 16])
def test_dependent_chain_eager_and_graph(oracle, M):
    x0, stages = make_chain(M)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        poison(stages)
        launch_chain(x0, stages)
    torch.cuda.synchronize()
    check_against_oracle(oracle, x0, stages, M)
    eager = [s["Y"].clone() for s in stages]

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        launch_chain(x0, stages)
    torch.cuda.synchronize()
    for rep in range(3):
        with torch.cuda.stream(stream):
            poison(stages)
            graph.replay()
        torch.cuda.synchronize()
        for i, (s, e) in enumerate(zip(stages, eager)):
            assert torch.equal(s["Y"].view(torch.int32), e.view(torch.int32)), f"replay {rep}, stage {i} differs"
    check_against_oracle(oracle, x0, stages, M)
    assert pnq.device_error() == 0
