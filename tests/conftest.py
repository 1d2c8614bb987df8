"""Shared pytest set-up: the repository root on sys.path and the ``gpu`` marker."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def orc():
    """The fp64 C oracle, compiled for this machine if needed."""
    import oracle

    if not os.path.exists(oracle.LIB) or os.path.getmtime(oracle.LIB) < os.path.getmtime(oracle.SRC):
        oracle.build()
    return oracle.Oracle()
