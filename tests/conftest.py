"""Shared pytest configuration: the ``gpu`` marker and small helpers."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


from tests.gpu_util import ops  # noqa: E402,F401  (session fixture for the GPU tests)
