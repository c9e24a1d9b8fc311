"""Shared pytest configuration: the ``gpu`` marker and small helpers."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size GPU parity case")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built C-ABI library (GPU tests only); fails loudly when it is missing."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected without a CUDA device")
    import mla_latent_kv_06_gb300 as mla
    mla.load()
    return mla
