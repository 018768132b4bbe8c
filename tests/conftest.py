import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload check")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="session")
def cuda():
    """Skip when no CUDA device is visible; otherwise make sure libmoe.so is built."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_ffn_19_b300 import build
    build.build()
    import mixture_experts_ffn_19_b300 as moe
    moe.lib()
    return torch.device("cuda:0")


def pytest_terminal_summary(terminalreporter):
    """Print the parity figures the GPU tests measured (norm-wise and element-wise
    error, near-ties and flips per case)."""
    try:
        from helpers import PARITY_REPORT
    except ImportError:
        return
    if not PARITY_REPORT:
        return
    tr = terminalreporter
    tr.section("parity report")
    for name, f in PARITY_REPORT:
        tr.write_line(name + ": " + ", ".join(
            f"{k} {v:.3g}" if isinstance(v, float) else f"{k} {v}" for k, v in f.items()))
