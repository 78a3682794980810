import importlib.util
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def build_library() -> str:
    """Compile the in-tree CUDA library if it is missing or stale (nvcc, no GPU needed)."""
    spec = importlib.util.spec_from_file_location(
        "hd_build", os.path.join(ROOT, "full_gqa_decode_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build()


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.load()


@pytest.fixture(scope="session")
def libpath():
    return build_library()


@pytest.fixture(scope="session")
def hd(libpath):
    import full_gqa_decode_gb300
    return full_gqa_decode_gb300
