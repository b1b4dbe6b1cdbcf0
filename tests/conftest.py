import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle

    return oracle.load()


def build_library():
    """Build libswiglu.so if it is missing or stale (loads the builder by path:
    importing the package needs the built library)."""
    import importlib.util

    path = os.path.join(ROOT, "gate_up_swiglu_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("_libswiglu_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build()
