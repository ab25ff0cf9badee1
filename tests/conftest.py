import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def lib_path():
    """Builds the C-ABI library if needed and returns its path (nvcc works without a GPU)."""
    from exact_attention_fa_gb300 import build
    return build.build_library()


@pytest.fixture(scope="session")
def cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_fa_gb300 import build
    build.build_library()
    return torch.device("cuda:0")
