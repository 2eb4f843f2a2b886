import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running check (large configurations)")


def gpu_available():
    try:
        import torch
    except ImportError:
        return False
    return torch.cuda.is_available()


@pytest.fixture(scope="session")
def fa_lib():
    """The built library via its binding; a GPU test that gets here without it fails."""
    if not gpu_available():
        pytest.fail("GPU test collected on a host without CUDA")
    from exact_attention_38_gb300 import fa

    return fa
