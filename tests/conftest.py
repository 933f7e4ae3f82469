import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the libdcp kernels)")
    config.addinivalue_line("markers", "slow: long-running case")
    # test modules import the libraries at collection time, so build them (if stale) before collecting
    import __graft_entry__
    __graft_entry__.build()


def has_gpu() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture
def gpu():
    if not has_gpu():
        pytest.skip("no CUDA device")
    import torch
    torch.cuda.set_device(0)
    return torch.device("cuda:0")
