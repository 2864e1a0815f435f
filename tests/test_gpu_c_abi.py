"""The C ABI from plain C: tests/c/abi_update.c is compiled with gcc against
include/grs.h, linked with libgrs.so, the CUDA runtime and the oracle, and
run; it exits 0 when the update matches the oracle."""
import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_update_from_plain_c(tmp_path):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from gradient_reduction_sharded_gb300 import _build
    import oracle
    lib = _build.build()
    olib = oracle.build()
    cuda = os.path.dirname(os.path.dirname(_build.nvcc()))
    exe = str(tmp_path / "abi_update")
    subprocess.check_call(["gcc", "-std=c11", "-O1", "-o", exe, os.path.join(ROOT, "tests", "c", "abi_update.c"),
                           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
                           lib, olib, "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm",
                           "-Wl,-rpath," + os.path.dirname(lib) + ":" + os.path.dirname(olib) + ":" +
                           os.path.join(cuda, "lib64")])
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.count(": ok") == 3, r.stdout
