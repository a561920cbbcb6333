"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every function
include/pnq.h declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

import block_quantized_weight_pn3t_gb300 as pnq
from block_quantized_weight_pn3t_gb300 import Status

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(pnq.lib_path()):
        from block_quantized_weight_pn3t_gb300 import build
        build.build()
    return pnq.lib()


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(pnq_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"pnq_gemv", "pnq_dequantize_row", "pnq_validate_row"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_version(lib):
    assert lib.pnq_version().decode().startswith("pnq")


FAKE = 0x10000  # never dereferenced: every call below fails its argument check first


@pytest.mark.parametrize("call", ["gemv", "dequantize", "validate"])
def test_argument_errors(lib, call):
    def run(type_, W, n, K, M=1, out=FAKE, X=FAKE):
        if call == "gemv":
            return pnq.gemv_ptr(type_, W, n, K, X, M, out)
        if call == "dequantize":
            return pnq.dequantize_row_ptr(type_, W, n, K, out)
        return pnq.validate_row_ptr(type_, W, n, K, out)

    assert run(7, FAKE, 4, 80) == Status.ERR_TYPE
    assert run(pnq.PN3T, FAKE, 4, 64) == Status.ERR_SHAPE       # not a multiple of 80
    assert run(pnq.PN4T, FAKE, 4, 80) == Status.ERR_SHAPE       # not a multiple of 64
    assert run(pnq.PN3T, FAKE, -1, 80) == Status.ERR_SHAPE
    assert run(pnq.PN3T, FAKE, 4, 0) == Status.ERR_SHAPE
    assert run(pnq.PN3T, 0, 4, 80) == Status.ERR_NULL
    assert run(pnq.PN3T, FAKE + 1, 4, 80) == Status.ERR_ALIGN   # W needs 2-byte alignment
    assert run(pnq.PN3T, FAKE, 4, 80, out=0) == Status.ERR_NULL
    assert run(pnq.PN3T, FAKE, 4, 80, out=FAKE + 2) == Status.ERR_ALIGN
    assert run(pnq.PN3T, FAKE, 0, 80) == Status.OK                # nothing to do, nothing launched
    assert run(pnq.PN3T, FAKE, 2 ** 62, 80 * 2 ** 20) == Status.ERR_SHAPE  # size overflow
    nv = pnq.nvfp4_weights(FAKE, FAKE, 0.01)
    assert run(pnq.NVFP4, nv, 4, 24) == Status.ERR_SHAPE          # K % 16
    assert run(pnq.NVFP4, pnq.nvfp4_weights(0, FAKE, 0.01), 4, 32) == Status.ERR_NULL
    assert run(pnq.NVFP4, pnq.nvfp4_weights(FAKE, 0, 0.01), 4, 32) == Status.ERR_NULL
    if call == "gemv":
        assert run(pnq.PN3T, FAKE, 4, 80, M=0) == Status.ERR_SHAPE
        assert run(pnq.PN3T, FAKE, 4, 80, M=17) == Status.ERR_SHAPE
        assert run(pnq.PN3T, FAKE, 4, 80, X=0) == Status.ERR_NULL
        assert run(pnq.PN3T, FAKE, 4, 80, X=FAKE + 2) == Status.ERR_ALIGN  # fp32 X
        assert run(pnq.NVFP4, nv, 4, 32, X=FAKE + 1) == Status.ERR_ALIGN   # bf16 X
        assert pnq.gemv_ex_ptr(pnq.PN3T, FAKE, 4, 80, FAKE, 1, FAKE, 2) == Status.ERR_FLAGS
        assert pnq.gemv_ex_ptr(pnq.PN3T, FAKE, 0, 80, FAKE, 1, FAKE, pnq.GEMV_STATIC_WEIGHTS) == Status.OK


def test_nvfp4_descriptor_null_pointer(lib):
    rc = lib.pnq_gemv(pnq.NVFP4, None, 4, 32, ctypes.c_void_p(FAKE), 1, ctypes.c_void_p(FAKE), None)
    assert rc == Status.ERR_NULL


def test_binding_raises_without_library(monkeypatch, tmp_path):
    from block_quantized_weight_pn3t_gb300 import _binding
    monkeypatch.setattr(_binding, "_lib", None)
    monkeypatch.setattr(_binding, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(pnq.PnqError):
        _binding.lib()


def test_wrappers_check_tensors_before_the_library(monkeypatch):
    """The torch wrappers pass only addresses, so they refuse a tensor of the wrong dtype, a
    non-contiguous one, one too small for the call, or a host tensor, before anything reaches
    the library."""
    import torch
    from block_quantized_weight_pn3t_gb300 import _binding

    def no_library():
        raise AssertionError("the library was called")
    monkeypatch.setattr(_binding, "lib", no_library)
    req = _binding._require
    with pytest.raises(pnq.PnqError, match="dtype"):
        req(torch.zeros(8, dtype=torch.float64), "X", (torch.float32,))
    with pytest.raises(pnq.PnqError, match="contiguous"):
        req(torch.zeros(4, 8, dtype=torch.float32).t(), "X", (torch.float32,))
    with pytest.raises(pnq.PnqError, match="elements"):
        req(torch.zeros(8, dtype=torch.float32), "Y", (torch.float32,), 9)
    with pytest.raises(pnq.PnqError, match="CUDA"):
        req(torch.zeros(8, dtype=torch.float32), "Y", (torch.float32,), 8)
    with pytest.raises(pnq.PnqError, match="torch.Tensor"):
        req([0.0] * 8, "Y", (torch.float32,))
    N, K = 4, 640
    W = torch.zeros(N * (K // 80) * 34, dtype=torch.uint8)
    with pytest.raises(pnq.PnqError, match="elements"):  # one byte short of 4 rows of pn3t
        pnq.gemv(pnq.PN3T, W[:-1], torch.zeros(1, K), N, K)
    with pytest.raises(pnq.PnqError, match="CUDA"):
        pnq.gemv(pnq.PN3T, W, torch.zeros(1, K), N, K)
    with pytest.raises(pnq.PnqError, match="CUDA"):
        pnq.dequantize_row(pnq.PN3T, W, N, K)
    with pytest.raises(pnq.PnqError, match="CUDA"):
        pnq.validate_row(pnq.NVFP4, (torch.zeros(N * 128, dtype=torch.uint8), torch.zeros(N * 16, dtype=torch.uint8),
                                     0.01), N, 256)


C_CLIENT = r"""
#include "pnq.h"
#include <stdio.h>
int main(void) {
    pnq_nvfp4_weights w = {0, 0, 0.01f};
    int32_t code = 0;
    int rc = pnq_gemv(PNQ_PN3T, 0, 0, 80, 0, 1, 0, (cudaStream_t)0);  /* N = 0: nothing launched */
    printf("%s|%d|%d|%d\n", pnq_version(), rc, (int)sizeof(w), PNQ_ERR_SCRATCH);
    (void)code; (void)pnq_device_error; (void)pnq_gemv_ex; (void)pnq_gemv_noalloc;
    (void)pnq_dequantize_row; (void)pnq_validate_row;
    return 0;
}
"""


def test_header_is_plain_c(lib, tmp_path):
    """include/pnq.h compiles as C99 and a C program links against libpnq.so and calls it."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if not gcc:
        pytest.skip("gcc not found")
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(pnq.lib_path())
    cuda_inc = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(shutil.which("nvcc") or
                                                                             "/usr/local/cuda/bin/nvcc"))), "include")
    subprocess.check_call([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), "-I",
                           cuda_inc, str(src), "-L", libdir, "-lpnq", f"-Wl,-rpath,{libdir}", "-o", str(exe)])
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    version, rc, size, scratch = out.stdout.strip().split("|")
    assert version.startswith("pnq ") and int(rc) == Status.OK and int(scratch) == Status.ERR_SCRATCH
    assert int(size) == ctypes.sizeof(pnq._binding.pnq_nvfp4_weights)
