"""The checked build (GRS_CHECKED=1): every kernel verifies each index it
derives against the extent of the buffer it addresses and records a failure
instead of making the access.  The GPU parity, robustness and checkpoint
suites run against that library in a child process; each plan's flags are
read when its test closes it, and no check may have fired.
"""
import os
import re
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_gpu_suites_pass_on_the_checked_build():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from gradient_reduction_sharded_gb300 import _build
    lib = _build.build_checked()
    probe = subprocess.run([sys.executable, "-c",
                            "from gradient_reduction_sharded_gb300 import grs; print(grs.grs_build_features())"],
                           cwd=ROOT, env=dict(os.environ, GRS_LIBRARY=lib), capture_output=True, text=True,
                           timeout=300)
    assert probe.returncode == 0 and probe.stdout.strip() == "1", probe.stdout + probe.stderr
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m",
                        "gpu and not slow", "tests/test_gpu_parity.py", "tests/test_gpu_robustness.py",
                        "tests/test_gpu_checkpoint.py"],
                       cwd=ROOT, env=dict(os.environ, GRS_LIBRARY=lib), capture_output=True, text=True,
                       timeout=1800)
    assert r.returncode == 0, (r.stdout[-4000:] + r.stderr[-2000:])
    m = re.search(r"(\d+) passed", r.stdout)
    assert m and int(m.group(1)) >= 30, r.stdout[-2000:]
