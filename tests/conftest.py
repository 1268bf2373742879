import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


def pytest_collection_modifyitems(config, items):
    # CPU-only runs on a machine without a GPU: a gpu-marked test is never
    # silently turned into a pass; it fails loudly if selected without a GPU.
    pass


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA C-ABI library through its Python binding (GPU tests only)."""
    import torch

    if not torch.cuda.is_available():
        pytest.fail("gpu test selected but no CUDA device is visible")
    from online_kv_cache_chunked_gb300 import binding

    binding.load()
    return binding
