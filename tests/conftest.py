"""Shared pytest configuration.

Tests marked ``gpu`` need a CUDA device and the compiled library; everything
else runs on the CPU (the oracle against its pins, host-side argument logic,
the workload generator and the library's exported symbols).
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the compiled libpnkv")
    config.addinivalue_line("markers", "slow: long CPU oracle run (full-size sampled checks)")


@pytest.fixture(scope="session")
def repo_root():
    return ROOT
