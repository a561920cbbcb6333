"""Host checks of the fast paths' launch logic, compiled for the CPU with nvcc (no GPU needed:
kernels are compiled but never launched):

- tests/host/split_check.cu: the cluster work split (csrc/pnq_split.cuh) and the launch planner
  (csrc/pnq_cluster.cuh) with the PN and NVFP4 format policies: row ranges and item shares tile
  the matrix, stage walks visit exactly a CTA's items, a row group always falls to one consumer
  warp, and every plan's shared-memory regions are disjoint, aligned and inside the budget it
  claims (two CTAs per SM, or one).
"""
import concurrent.futures
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "block_quantized_weight_pn3t_gb300", "csrc")
HOST = os.path.join(ROOT, "tests", "host")
CHECKS = {"split_check": 60000}  # least count expected


def nvcc():
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        pytest.skip("nvcc not found")
    return path


@pytest.fixture(scope="module")
def runs(tmp_path_factory):
    nv = nvcc()
    out = tmp_path_factory.mktemp("host_checks")

    def build_and_run(name):
        exe = str(out / name)
        # PTX only (no ptxas): nothing runs on a GPU
        subprocess.check_call([nv, "-gencode", "arch=compute_103a,code=compute_103a", "-O2", "-std=c++17",
                               "--expt-relaxed-constexpr", "-I", CSRC, "-I", os.path.join(ROOT, "include"), "-I",
                               HOST, os.path.join(HOST, name + ".cu"), "-o", exe])
        return name, subprocess.run([exe], capture_output=True, text=True, timeout=600)

    with concurrent.futures.ThreadPoolExecutor(len(CHECKS)) as ex:
        return dict(ex.map(build_and_run, CHECKS))


@pytest.mark.parametrize("name", list(CHECKS))
def test_host_check(runs, name):
    r = runs[name]
    assert r.returncode == 0 and r.stdout.startswith("ok "), r.stdout[-2000:] + r.stderr[-2000:]
    assert int(r.stdout.split()[1]) >= CHECKS[name]  # configurations or plans checked
