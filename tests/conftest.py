import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libkl.so")
    config.addinivalue_line("markers", "slow: full-size parity runs")


@pytest.fixture(scope="session")
def kl():
    """The CUDA library binding; GPU tests only."""
    import torch

    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without CUDA")
    import bwd_qwen3_layer_gb300 as k

    k.load()
    return k
