import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libpstat.so")


@pytest.fixture(scope="session")
def cuda_lib():
    """The C-ABI library, built for the GPU that runs the tests."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from vocab_wide_token_gb300 import pstat

    return pstat
