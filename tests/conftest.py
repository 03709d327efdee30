import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


@pytest.fixture(autouse=True)
def _checked_build_reports_no_violation(request):
    """Under FUSEDWIN_CHECKED=1 (the bounds-checked library), every GPU test must
    leave the device error words clear: no kernel touched memory outside a buffer."""
    yield
    if os.environ.get("FUSEDWIN_CHECKED") == "1" and request.node.get_closest_marker("gpu"):
        from pooling_sliding_window_gb300 import fusedwin as FW
        FW.fw_check_device_errors()  # raises FusedWinError unless FW_OK
