"""Shared pytest configuration.

Markers:
  gpu  -- needs a CUDA device (a GB300, sm_103); everything else runs on CPU.
"""
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
    config.addinivalue_line("markers", "gpu: test needs a CUDA device (sm_103)")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.get()
