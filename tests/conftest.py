"""Shared pytest configuration.

``-m gpu`` tests run the CUDA library on a GB300; everything else runs on a
CPU-only host (the oracle and its pins, host logic, the C-ABI symbol table).
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def oracle():
    import oracle as oracle_pkg

    return oracle_pkg.load()
