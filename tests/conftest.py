import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def gpu_lib():
    """The loaded C-ABI library; only for tests marked gpu."""
    import torch

    if not torch.cuda.is_available():
        pytest.fail("gpu test run without a CUDA device")
    from kv_cache_quantization_append_gb300 import lib

    return lib.load()
