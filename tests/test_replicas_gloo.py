"""The multi-process path of bench.py on CPU: two ranks over gloo (127.0.0.1).

The GEMV shards by output rows with no exchange, so N > 1 runs independent replicas of the step;
the only cross-rank steps are the slowest-rank time and rank 0 alone reporting. These run here as
world_size-2 gloo process groups (no GPU)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, os, sys
sys.path.insert(0, {root!r})
import torch.distributed as dist
dist.init_process_group("gloo", init_method="tcp://127.0.0.1:{port}", rank={rank}, world_size=2)
import bench
times = [10.0 + {rank}, 20.0 - 3 * {rank}]  # rank 1 is slower on the first, faster on the second
slowest, gbps = bench.aggregate_replicas(times, 2, 4e9, dist)
dist.barrier()
print(json.dumps({{"rank": {rank}, "slowest": slowest, "gbps": gbps}}))
dist.destroy_process_group()
"""


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def run_ranks(script, env=None, timeout=120):
    procs = [subprocess.Popen([sys.executable, "-c", script(r)], stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                              text=True, env=env) for r in range(2)]
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=timeout)
        assert p.returncode == 0, err[-3000:]
        outs.append(out)
    return outs


def test_slowest_rank_and_whole_job_bytes():
    port = free_port()
    outs = run_ranks(lambda r: CHILD.format(root=ROOT, port=port, rank=r))
    for r, out in enumerate(outs):
        res = json.loads(out.strip().splitlines()[-1])
        assert res["rank"] == r
        assert res["slowest"] == [11.0, 20.0]  # max over ranks, element by element
        # bytes of both replicas over the slowest rank's time
        assert res["gbps"] == pytest.approx([2 * 4e9 / 11e-3 / 1e9, 2 * 4e9 / 20e-3 / 1e9])


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    slowest, gbps = bench.aggregate_replicas([5.0], 1, 1e9, None)
    assert slowest == [5.0] and gbps == pytest.approx([200.0])


def test_reference_arm_prints_on_rank_0_only():
    """Under torchrun the reference arm (the oracle on the host cores) runs on rank 0 alone; the
    other ranks exit 0 without work or output."""
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    assert r.stdout.strip() == ""


def test_reference_arm_line_matches_our_config():
    """Rank 0's reference line: the contract's keys, the same workload `config` our arm reports
    (plus how it was sampled), and e2e with no host-device bytes."""
    sys.path.insert(0, ROOT)
    import bench
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--layers", "2"], env=env, capture_output=True, text=True, timeout=300,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == "GB/s"
    assert line["higher_is_better"] is True and line["value"] > 0
    ours = bench.workload_config(1, 2, 2 * len(bench.PROJECTIONS), 1)
    assert {k: v for k, v in line["config"].items() if k != "sample"} == ours
    assert ours["weight_bytes_per_step"] == 2 * 172_130_304
    assert line["cpu_baseline"]["value"] == line["value"] and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
