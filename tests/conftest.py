import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA path through the C ABI)")
    config.addinivalue_line("markers", "slow: long-running oracle case")


@pytest.fixture(scope="session")
def lib():
    """The C-ABI library, loaded through the thin Python binding (GPU tests only)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from recoverable_quantized_kv_gb300 import binding
    return binding.load()
