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
def lynx_lib():
    """Builds (if needed) and loads the in-tree CUDA library."""
    from progressive_kv_quantization_gb300 import build as _build
    from progressive_kv_quantization_gb300 import lynx as _lynx
    _build.build()
    return _lynx.load()


@pytest.fixture(scope="session")
def cuda_device(lynx_lib):
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for tests marked gpu")
    torch.cuda.init()
    return torch.device("cuda:0")
