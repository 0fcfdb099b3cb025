import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle_mod():
    from oracle import oracle
    oracle.lib()
    return oracle


@pytest.fixture(autouse=True)
def _debug_build_bounds_check(request):
    """With the bounds-checking debug library (RMSQ_DEBUG=1), no GPU test may
    leave a failed store check behind in the status word."""
    yield
    if os.environ.get("RMSQ_DEBUG") == "1" and request.node.get_closest_marker("gpu"):
        from mxfp4_activation_quant_gb300 import rmsq
        assert rmsq.sync_status() == 0, "a debug-build bounds check failed (or a wait timed out)"
