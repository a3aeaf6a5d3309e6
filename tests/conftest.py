import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built liblossk.so")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


def build_lib():
    """Build liblossk.so (loading build.py by path; the package import needs the library)."""
    import importlib.util
    path = os.path.join(ROOT, "output_projection_cross_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("lossk_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build()
