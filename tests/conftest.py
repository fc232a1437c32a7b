"""Test configuration: the `gpu` marker and import paths.

`-m "not gpu"` runs the oracle pins, host-side logic and the C-ABI symbol checks on a
machine without a GPU; `-m gpu` runs the parity tests through the C ABI on one GPU.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running parity sweep")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")
