import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a)")


def pytest_collection_modifyitems(config, items):
    # A gpu test on a machine without CUDA is an error, not a skip: the driver
    # runs "-m gpu" only on GPU machines, and a silent skip there would hide a
    # missing native path.
    pass


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")
