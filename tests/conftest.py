import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


@pytest.fixture(scope="session")
def gb():
    """The CUDA library through its Python binding (GPU tests only)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_fp16_flashattention_gb300 as pkg
    pkg.load()
    pkg.set_wait_limit_ns(1_000_000_000)   # in-kernel waits give up after 1 s
    return pkg
