import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: large CPU oracle work")


@pytest.fixture(scope="session")
def gpu_lib():
    """The CUDA library through its Python binding; skips only when no GPU exists."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import layer_streamed_qlora_linear_b300 as sl
    return sl
