import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built C-ABI library on a machine with a CUDA GPU; GPU tests fail loudly without it."""
    import torch
    import exact_tiled_attention_21_gb300 as fa
    assert torch.cuda.is_available(), "GPU test run without a CUDA device"
    fa.load()  # raises if the shared library is missing
    return fa
