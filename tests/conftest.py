"""Shared test setup: the repository root on sys.path and the ``gpu`` marker.

Tests marked ``gpu`` need a GB300 (sm_103) and the CUDA library built for it;
everything else runs on CPU in a few minutes.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 GPU and the CUDA library")
    config.addinivalue_line("markers", "slow: K3-sized case (minutes)")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")
