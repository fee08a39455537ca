import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def lq():
    """The package with liblq.so built (in-tree) and loaded."""
    from gemm_gemv_f16w_gb300 import build as b
    b.build()
    import gemm_gemv_f16w_gb300 as pkg
    pkg.lib()
    return pkg


@pytest.fixture(scope="session")
def cuda_dev(lq):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    return torch.device("cuda:0")
