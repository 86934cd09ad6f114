"""Shared pytest setup: repo root on sys.path and the ``gpu`` marker.

Tests marked ``gpu`` need a CUDA device of compute capability 10.3 and the
built ``libmgattn.so``; everything else runs on a CPU-only machine.
"""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a compute-capability 10.3 GPU and libmgattn.so")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle

    return oracle.load_library()
