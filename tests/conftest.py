import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs on the GB300 box)")
    config.addinivalue_line("markers", "slow: long-running parity case")


@pytest.fixture(scope="session")
def libuocr():
    """Build (if stale) and load the CUDA library."""
    from quantized_moe_decode_gb300 import binding, build

    build.build()
    return binding.load()


@pytest.fixture(scope="session")
def cuda(libuocr):
    import torch

    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for -m gpu tests")
    torch.cuda.init()
    return torch
