import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA device (GB300, sm_103a) and the built library")


@pytest.fixture(scope="session")
def lib():
    """The built C-ABI library through its Python binding (GPU tests only)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_paged_kv_varlen_gb300 as q
    if not os.path.exists(q.LIB_PATH):
        from quantized_paged_kv_varlen_gb300 import build
        build.build()
    q.load()
    return q
