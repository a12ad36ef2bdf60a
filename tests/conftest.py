import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size parity case (minutes of oracle time)")


@pytest.fixture(scope="session")
def lmh():
    """The CUDA library's Python binding, on a GPU machine (build it if needed)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_reduction_gb300 import _build
    _build.build()
    import top_reduction_gb300 as pkg
    return pkg
