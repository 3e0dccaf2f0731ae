"""Shared pytest setup: markers and import paths."""
import sys
from pathlib import Path

REPO = Path(__file__).resolve().parent.parent
for p in (REPO, REPO / "tests"):
    if str(p) not in sys.path:
        sys.path.insert(0, str(p))


import pytest


@pytest.fixture
def test_build():
    """Route the test's library calls to the test build, which honours the
    SS_NCHUNKS / SS_CTAS_PER_SM plan overrides, SS_MAMBA2_ROWS and SS_TEST_SKIP_UNITS."""
    import mamba_selective_scan_ss_gb300 as ss
    with ss.test_hooks():
        yield


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
