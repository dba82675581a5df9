import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running full-size case")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


def pytest_sessionfinish(session, exitstatus):
    """Under the store-checked library (TIDE_LIBRARY=checked), write the
    number of stores the kernels skipped to the file TIDE_BOUNDS_REPORT names."""
    report = os.environ.get("TIDE_BOUNDS_REPORT")
    if report and os.environ.get("TIDE_LIBRARY") == "checked":
        import fsdp_layout_aware_gb300 as tide
        with open(report, "w") as f:
            f.write(str(tide.tide_debug_bounds_violations()))
