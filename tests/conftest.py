"""Shared pytest configuration.

Tests marked ``gpu`` need a CUDA device and the built library; everything else
runs on the CPU alone.
"""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300) and the built library")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built library and binding, on a CUDA device; fails loudly if missing."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("gpu test collected on a machine without a CUDA device")
    import fp8_fine_grained_19_b300 as fp8
    fp8.load()
    return fp8
