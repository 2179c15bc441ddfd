import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA library through its C ABI)")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library's Python binding, built in-tree; skips without a GPU."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import compressed_sparse_decode_gb300 as csd
    csd.load()
    return csd
