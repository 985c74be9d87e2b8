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
    config.addinivalue_line("markers", "gpu: needs an sm_103 GPU and the built CUDA library")


@pytest.fixture(scope="session")
def sage_lib():
    """The CUDA library loaded through the Python binding (built on demand)."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_attention_fp64_gb300 import _lib

    _lib.ensure_built()
    return _lib.load()
