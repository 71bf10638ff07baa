"""Failure detection on the GPU without a fault: device-side waits that nothing satisfies
give up after their limit, report HYB_DEVERR_TIMEOUT through the device status word, and
leave the context usable for the next call."""
import time

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import assert_out_close, assert_states_close, empty_rows, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_us", [2000, 50000])
def test_bounded_waits_expire_report_and_return(hyb, devstatus, limit_us):
    t0 = time.perf_counter()
    hyb.check(hyb.hyb_selftest_bounded_waits(limit_us))
    torch.cuda.synchronize()
    took = time.perf_counter() - t0
    st, flags = hyb.hyb_device_status(clear=True)
    assert st == hyb.HYB_ERR_DEVICE_CHECK
    assert flags == hyb.HYB_DEVERR_TIMEOUT
    assert took >= limit_us * 1e-6                   # the waits ran to their limit ...
    assert took < limit_us * 1e-6 + 5.0              # ... and then returned

    # the context is still usable: a linear decode step runs and matches the oracle
    g = W.rng(5)
    B, H, D, NS = 3, 4, 64, 5
    q, k, v = (W.rows(g, (B, H, D), D, W.BF16) for _ in range(3))
    pool = W.synthetic_state(g, NS, H, D, np.full(NS, 100))
    slots = np.array([4, 0, 2], np.int32)
    o_ref, s_ref = oracle.linear_step(q, k, v, pool, slots)
    pool_d = to_dev(pool)
    out = empty_rows((B, H, D), W.BF16)
    hyb.check(hyb.hyb_linear_attn_step(out, to_dev(q), to_dev(k), to_dev(v), pool_d, NS, to_dev(slots),
                                       B, H, D, W.BF16))
    torch.cuda.synchronize()
    assert_out_close(out, o_ref, "linear step after the self-test")
    assert_states_close(to_host(pool_d)[slots], s_ref, "states after the self-test")
    assert devstatus() == (0, 0)
