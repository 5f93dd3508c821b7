import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs on the GB300 box)")
    config.addinivalue_line("markers", "slow: full-size cases (minutes)")


def gpu_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library, built in-tree. A GPU test never runs without it."""
    if not gpu_available():
        pytest.fail("gpu test selected but no CUDA device is visible")
    import paged_kv_attention_pa_gb300 as pa
    pa.load()  # raises if the shared library is missing
    return pa


def pytest_terminal_summary(terminalreporter):
    """The largest error against the float64 oracle that any parity check measured."""
    try:
        from harness import RECORDED
    except Exception:
        return
    if not RECORDED:
        return
    what, err = max(RECORDED, key=lambda x: x[1])
    terminalreporter.write_line(
        f"parity: {len(RECORDED)} comparisons with the float64 oracle; largest rel L-inf "
        f"error {err:.3e} ({what})")
