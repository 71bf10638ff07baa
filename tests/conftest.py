import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libhyb.so")


import pytest  # noqa: E402


@pytest.fixture(scope="session")
def hyb():
    """The libhyb.so binding, built in-tree first if stale. GPU tests skip without CUDA."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_linear_gb300 import _build
    _build.build()
    import paged_kv_linear_gb300 as hyb_mod
    st, flags = hyb_mod.hyb_device_status(clear=True)
    assert st in (0, hyb_mod.HYB_ERR_DEVICE_CHECK)
    return hyb_mod


@pytest.fixture()
def devstatus(hyb):
    """Clears the device status word before a test; yields a reader (status, flags)."""
    hyb.hyb_device_status(clear=True)
    yield lambda: hyb.hyb_device_status(clear=True)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Worst achieved row-relative output error per test (the parity margin of each check)."""
    try:
        from gpu_helpers import RECORDS, ROW_REL
    except ImportError:
        return
    if not RECORDS:
        return
    worst = {}
    for tid, what, rel, abs_err in RECORDS:
        if tid not in worst or rel > worst[tid][1]:
            worst[tid] = (what, rel, abs_err)
    tr = terminalreporter
    tr.write_sep("-", f"output parity: worst row-relative error per test (bound {ROW_REL:g})")
    for tid, (what, rel, abs_err) in sorted(worst.items(), key=lambda kv: -kv[1][1]):
        tr.write_line(f"{rel:.2e}  abs {abs_err:.2e}  {tid}  [{what}]")
