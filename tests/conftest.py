import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def load_golden(name):
    import json
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.get()


def build_library():
    """Compile the CUDA library (loading the build script by path, so that the
    package itself is imported only once the library exists)."""
    import importlib.util
    path = os.path.join(ROOT, "spmv_sparse_storage_gb300", "_build.py")
    spec = importlib.util.spec_from_file_location("_spmv_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build()
