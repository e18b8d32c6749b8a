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


def pytest_terminal_summary(terminalreporter):
    """The rounding-edge code fraction over every GPU code comparison of the run
    (codes may differ from the oracle's by +-1 only within 1e-5 of an edge, and
    that fraction must stay below 1e-4)."""
    import lynx_testutil
    if lynx_testutil.CODE_TALLY:
        n = sum(d for d, _ in lynx_testutil.CODE_TALLY)
        tot = sum(c for _, c in lynx_testutil.CODE_TALLY)
        worst = max(d / c for d, c in lynx_testutil.CODE_TALLY)
        terminalreporter.write_line(f"rounding-edge +-1 codes: {n} of {tot} compared ({n / tot:.3g}); "
                                    f"largest fraction in one check {worst:.3g} (bar 1e-4)")
