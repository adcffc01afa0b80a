import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) GPU and the CUDA library")


def has_gb300() -> bool:
    try:
        import torch
        if not torch.cuda.is_available():
            return False
        major, minor = torch.cuda.get_device_capability(0)
        return (major, minor) == (10, 3)
    except Exception:
        return False


@pytest.fixture(scope="session")
def gpu():
    """Skip-free guard: a test marked gpu fails loudly (rather than skipping)
    when run without the GPU it needs."""
    import torch
    assert torch.cuda.is_available(), "this test needs a CUDA GPU"
    assert torch.cuda.get_device_capability(0) == (10, 3), "this test needs an sm_103 GPU"
    return torch.device("cuda:0")
