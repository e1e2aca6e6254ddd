import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (sm_103a); parity tests of the CUDA path")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def cuda_device():
    """The CUDA device for parity tests.  A missing GPU or a missing library is
    an error, never a skip: the CUDA path has no fallback."""
    import torch
    if not torch.cuda.is_available():
        raise RuntimeError("gpu-marked test run without a CUDA device")
    import block_quantized_weight_qp_gb300 as qp
    qp.load()
    return torch.device("cuda:0")
