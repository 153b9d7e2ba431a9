"""Shared pytest setup: the ``gpu`` marker and small fixtures.

Tests marked ``gpu`` need a CUDA device and the compiled CUDA library; every
other test runs on the CPU only (the oracle, its pins, host-side argument
checks of the C ABI and the multi-process host logic).
"""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the compiled CUDA library")


@pytest.fixture(scope="session")
def cuda_lib():
    """The product library, loaded through its Python binding (GPU tests only)."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    import dlrm_embeddings_dot_gb300 as dl
    dl.load()
    return dl
