import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def golden_path(name: str) -> str:
    return os.path.join(ROOT, "tests", "golden", name)


@pytest.fixture(scope="session")
def built_lib_path():
    """Path of the compiled C-ABI library, building it if it is missing."""
    from rotated_bit_kv_kvq_gb300 import build as kbuild
    return kbuild.ensure_built()
