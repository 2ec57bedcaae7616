import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built afx library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds")


@pytest.fixture(scope="session")
def golden_dir():
    return GOLDEN


DEBUG_BOUNDS = os.environ.get("AFX_DEBUG_BOUNDS", "0") == "1"


@pytest.fixture(scope="session")
def afx():
    """The product binding, built in-tree first if needed (nvcc cross-compiles
    here).  With AFX_DEBUG_BOUNDS=1 it is the bounds-checked build, and the
    session fails at its end if any kernel's bounds check fired."""
    from weight_streaming_canonical_gb300 import build as _build
    _build.build(debug_bounds=DEBUG_BOUNDS)
    from weight_streaming_canonical_gb300 import afx as _afx
    yield _afx
    if DEBUG_BOUNDS:
        bits, checked = _afx.afx_debug_bounds_report()
        assert checked, "AFX_DEBUG_BOUNDS=1 but the loaded library does not check bounds"
        assert bits == 0, f"bounds checks failed during the session: {bits:#x}"
