import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    # keep the order files are collected in (test_zz_* last), tests inside a
    # file in definition order
    pass


@pytest.fixture(scope="session")
def cuda_lib():
    """The built C-ABI library (built in-tree if missing)."""
    from radixattention_prefix_shared_gb300 import binding
    return binding.lib()
