"""State-precision study on the GPU: the linear decode step over a 16-bit (bf16 / fp16)
state pool against the CPU oracle's 16-bit recurrence (states bit for bit), and the drift
that 16-bit states cause against the fp64 recurrence, compared with the fp32 state the
pages prescribe."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import as_f64, assert_out_close, empty_rows, to_dev, to_host

pytestmark = pytest.mark.gpu

F16 = 2


def _round16(x32, state_dtype):
    """fp32 -> 16-bit bit patterns (round to nearest even) by torch / numpy."""
    x32 = np.ascontiguousarray(x32, dtype=np.float32)
    if state_dtype == W.BF16:
        return torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return x32.astype(np.float16).view(np.uint16)


def _steps(hyb, q, k, v, cu, steps, state_dtype, pool_h, slots_h, dtype):
    """Runs `steps` decode steps (token s of every request per step) on the GPU; returns
    the outputs [B*steps][H][D] in packed order and the final pool."""
    B = len(cu) - 1
    H, D = q.shape[1], q.shape[2]
    pool = to_dev(pool_h)
    slots = to_dev(slots_h)
    outs = np.zeros(q.shape, np.float64)
    for s in range(steps):
        rows = np.asarray(cu[:-1]) + s
        qs, ks, vs = to_dev(q[rows]), to_dev(k[rows]), to_dev(v[rows])
        out = empty_rows((B, H, D), dtype)
        if state_dtype == W.F32:
            hyb.check(hyb.hyb_linear_attn_step(out, qs, ks, vs, pool, pool_h.shape[0], slots, B, H, D, dtype))
        else:
            hyb.check(hyb.hyb_linear_attn_step_lowp(out, qs, ks, vs, pool, state_dtype, pool_h.shape[0], slots,
                                                    B, H, D, dtype))
        outs[rows] = as_f64(out)
    torch.cuda.synchronize()
    return outs, to_host(pool)


@pytest.mark.parametrize("state_dtype", [W.BF16, F16])
@pytest.mark.parametrize("dtype,D", [(W.BF16, 128), (W.F32, 64)])
def test_lowp_step_states_bit_exact_with_oracle(hyb, devstatus, state_dtype, dtype, D):
    B, H, steps = 4, 4, 8
    g = W.rng(500 + D + state_dtype)
    cu = W.cu_from_lens(np.full(B, steps, np.int32))
    q, k, v = (W.rows(g, (B * steps, H, D), D, dtype) for _ in range(3))
    st0 = W.synthetic_state(g, B + 2, H, D, np.full(B + 2, 1000))
    pool_h = _round16(st0, state_dtype)                  # 2 slots more than requests
    slots_h = g.permutation(B + 2)[:B].astype(np.int32)
    outs, pool = _steps(hyb, q, k, v, cu, steps, state_dtype, pool_h, slots_h, dtype)
    ref_out, ref_st = oracle.linear_recurrence_lowp(q, k, v, cu, state_dtype, state_pool=pool_h,
                                                    state_slots=slots_h)
    assert np.array_equal(pool[slots_h], ref_st)         # fmaf + one rounding: same bits
    untouched = np.setdiff1d(np.arange(B + 2), slots_h)
    assert np.array_equal(pool[untouched], pool_h[untouched])
    assert_out_close(outs, ref_out, "16-bit-state step")
    assert devstatus() == (0, 0)


def test_state_precision_drift(hyb, devstatus):
    """2048 decode steps from a zero state (B=2, H=2, D=128, fp32 q/k/v and outputs, so no
    output rounding hides the state's): outputs against the fp64 recurrence. The fp32
    state stays at fp32 rounding level; 16-bit states drift far more (bf16 most: updates
    below half a spacing are lost), and their GPU states equal the oracle's 16-bit
    recurrence bit for bit after all 2048 steps."""
    B, H, D, steps = 2, 2, 128, 2048
    g = W.rng(520)
    cu = W.cu_from_lens(np.full(B, steps, np.int32))
    q, k, v = (W.rows(g, (B * steps, H, D), D, W.F32) for _ in range(3))
    slots_h = np.arange(B, dtype=np.int32)
    ref, _ = oracle.linear_recurrence(q, k, v, cu)
    last = np.concatenate([np.arange(cu[b + 1] - 64, cu[b + 1]) for b in range(B)])
    scale = np.abs(ref[last]).max()
    err = {}
    for sd in (W.F32, W.BF16, F16):
        pool_h = np.zeros((B, H, D, D), np.float32) if sd == W.F32 else np.zeros((B, H, D, D), np.uint16)
        outs, pool = _steps(hyb, q, k, v, cu, steps, sd, pool_h, slots_h, W.F32)
        err[sd] = float(np.abs(outs[last] - ref[last]).max() / scale)
        if sd != W.F32:
            _, ref_st = oracle.linear_recurrence_lowp(q, k, v, cu, sd)
            assert np.array_equal(pool, ref_st)
    print(f"relative output error after {steps} steps: fp32 {err[W.F32]:.2e}, bf16 {err[W.BF16]:.2e}, "
          f"fp16 {err[F16]:.2e}")
    assert err[W.F32] < 1e-4
    assert err[F16] > 10 * err[W.F32] and err[W.BF16] > err[F16]
    assert devstatus() == (0, 0)
