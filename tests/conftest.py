import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workloads")


@pytest.fixture(scope="session")
def cuda_lib():
    """Build and load the CUDA library; GPU tests need a device."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_attention_sage_gb300 as qas

    qas.build()
    return qas
