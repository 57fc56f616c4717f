import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def golden_dir():
    return GOLDEN


def _ensure_library_built():
    """Builds librf_gb300.so if it is missing or older than its sources (a no-op
    otherwise), so that every test sees the library of the current sources."""
    import __graft_entry__

    __graft_entry__._load_build_module().build()


_ensure_library_built()
