import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


def gpu_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA path's Python binding, built and loaded (GPU tests only)."""
    if not gpu_available():
        pytest.skip("no CUDA device")
    import variable_length_prefill_gb300 as vlp
    vlp.load()
    return vlp


def pytest_sessionfinish(session, exitstatus):
    """Write the parity errors of this run to $ATTN_VARLEN_REPORT_DIR, if set."""
    try:
        from gpu_helpers import REPORT
    except Exception:
        return
    out = os.environ.get("ATTN_VARLEN_REPORT_DIR")
    if not REPORT or not out or not os.path.isdir(out):
        return
    with open(os.path.join(out, "parity_report.txt"), "w") as f:
        f.write("case elements max_abs_err mean_abs_err\n")
        for what, n, mx, mean in REPORT:
            f.write(f"{what} {n} {mx:.3e} {mean:.3e}\n")
