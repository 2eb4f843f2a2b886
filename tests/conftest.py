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


def pytest_terminal_summary(terminalreporter):
    """How many compared elements exceeded the flat max-abs figure (the bound the tests
    apply adds half a unit in the last place of the output format at the reference)."""
    try:
        from _parity import FLAT_EXCESS
    except ImportError:
        return
    if not FLAT_EXCESS:
        return
    n = sum(c for _, c, _, _ in FLAT_EXCESS)
    tot = sum(t for _, _, t, _ in FLAT_EXCESS)
    terminalreporter.write_line(
        f"parity: {n} of {tot} elements in {len(FLAT_EXCESS)} comparisons exceeded the flat max-abs figure "
        f"(all within it plus half an output ulp); largest |ref| among them "
        f"{max(r for _, _, _, r in FLAT_EXCESS):.3f}")
    for name, c, t, r in sorted(FLAT_EXCESS, key=lambda e: -e[1])[:10]:
        terminalreporter.write_line(f"  {name}: {c} of {t} (max |ref| {r:.3f})")
