"""Host check of the stream-K work split the tensor-core GEMV kernels share (Sched in
csrc/pnq_streamk.cuh): tests/host/sched_check.cu is compiled for the CPU with nvcc and walks the
items of many (row tiles, K units, grid, item order) configurations, checking the item
bijection, the CTA shares, each tile's partial-share count (the tile counter's target), the
workspace slots the finishing CTA reads, and the resident operand span against brute force.
No GPU is needed: only host code runs."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "block_quantized_weight_pn3t_gb300", "csrc")


def nvcc():
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        pytest.skip("nvcc not found")
    return path


def test_work_split_against_brute_force(tmp_path):
    exe = str(tmp_path / "sched_check")
    subprocess.check_call([nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                           "--expt-relaxed-constexpr", "-I", CSRC, "-I", os.path.join(ROOT, "include"),
                           os.path.join(ROOT, "tests", "host", "sched_check.cu"), "-o", exe])
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.startswith("ok "), r.stdout[-2000:]
    assert int(r.stdout.split()[1]) > 5000  # configurations checked
