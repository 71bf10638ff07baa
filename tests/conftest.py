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
