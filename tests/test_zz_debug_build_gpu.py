"""The bounds-checking debug build (RMSQ_DEBUG): every global store of the
kernels checks its index against the output's extent and records a failure
in the status word (RMSQ_ERR_BOUNDS) instead of trapping -- the stand-in for a
memory checker. The parity, GEMM and randomized suites run against it in a
child process, which checks the status word after every GPU test."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_suites_pass_on_the_bounds_checking_build():
    from mxfp4_activation_quant_gb300 import build
    build.build(debug=True)
    env = dict(os.environ, RMSQ_DEBUG="1")
    suites = ["tests/test_random_gpu.py", "tests/test_gemm_gpu.py", "tests/test_parity_gpu.py"]
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", *suites], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert "passed" in r.stdout
