import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (GB300, sm_103a); parity against "
        "the oracle through the C ABI")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(autouse=True)
def _no_failed_bounds_check(request):
    """Under the bounds-checked debug build (VT_CHECKS=1), every GPU test
    ends by asserting that no device bounds check failed during it."""
    yield
    if (os.environ.get("VT_CHECKS", "") == "1"
            and request.node.get_closest_marker("gpu") is not None):
        import torch
        import frequency_ranked_drafter_gb300 as vt
        torch.cuda.synchronize()
        line = vt.load().vt_debug_checks()
        assert line == 0, f"a device bounds check failed (source line {line})"
