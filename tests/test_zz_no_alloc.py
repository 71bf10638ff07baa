"""The allocation-free paged decode entry point (collected last on purpose).

hyb_paged_attn_decode_noalloc serves callers that cannot allocate device memory -- for
example a runtime that plans all device memory itself and hands an op nothing but its
inputs and outputs, or a latency-critical loop that must not call cudaMalloc because it
synchronises the device. Its split-K partials live in a fixed 16 MiB array owned by the
library instead of a caller workspace. Here it is called through the C ABI twice in a
row, on two different batches. It runs the same kernels with the same split plan as
hyb_paged_attn_decode (with a caller workspace), so each result must equal that entry
point's bit for bit; the second call also shows that what the first call left in the
shared array does not leak into the next result. A third batch with peaked scores is
checked against the CPU oracle under the output rule the parity tests use.
"""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import assert_out_close, decode_case, to_dev, to_host

pytestmark = pytest.mark.gpu


def _batch(seed, lens, H=32, D=128):
    g = W.rng(seed)
    lens = np.asarray(lens, np.int32)
    pool = W.block_pool(g, lens)
    kc = W.device_rows_(torch.empty((pool.num_blocks, H, 16, D), dtype=torch.bfloat16, device="cuda"), seed + 1, D)
    vc = W.device_rows_(torch.empty_like(kc), seed + 2, D)
    q = to_dev(W.rows(g, (len(lens), H, D), D, W.BF16))
    return dict(lens=lens, pool=pool, kc=kc, vc=vc, q=q, H=H, D=D)


def _both(hyb, b):
    B, H, D = len(b["lens"]), b["H"], b["D"]
    d = hyb.dims(H, D, b["pool"].num_blocks, b["pool"].max_blocks, W.BF16)
    msl = int(b["lens"].max())
    bt, lens = to_dev(b["pool"].block_tables), to_dev(b["lens"])
    ws_n = hyb.hyb_paged_attn_decode_workspace_size(B, msl, d)
    assert 0 < ws_n <= 16 << 20
    ws = torch.empty(ws_n, dtype=torch.uint8, device="cuda")
    ref = torch.empty((B, H, D), dtype=torch.bfloat16, device="cuda")
    got = torch.full_like(ref, float("nan"))
    hyb.check(hyb.hyb_paged_attn_decode(ref, b["q"], b["kc"], b["vc"], bt, lens, B, msl, d, ws, ws_n))
    hyb.check(hyb.hyb_paged_attn_decode_noalloc(got, b["q"], b["kc"], b["vc"], bt, lens, B, msl, d))
    torch.cuda.synchronize()
    return got, ref


def test_noalloc_decode_equals_workspace_decode_on_two_calls_in_a_row(hyb):
    first = _batch(41, [4096, 17, 1500, 3000, 640, 2222, 9, 4000])
    second = _batch(42, [3500, 2048, 100, 4095, 1, 2900])
    for b in (first, second):
        got, ref = _both(hyb, b)
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))   # same kernels, same plan
    st, flags = hyb.hyb_device_status(clear=True)
    assert st == 0, f"device status {flags:#x}"


def test_noalloc_decode_matches_oracle_on_peaked_scores(hyb):
    """Rising scores: the running max moves across every split, so the merge of the splits'
    partials from the shared array must weight them right."""
    c = decode_case(43, [4096, 513, 9000, 1], 8, 128, W.BF16, peaked="rise")
    d = c.dims(hyb)
    lens = c.ctx + 1
    out = torch.full((c.B, c.H, c.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    hyb.check(hyb.hyb_paged_attn_decode_noalloc(out, to_dev(c.q), to_dev(c.okc), to_dev(c.ovc),
                                                to_dev(c.pool.block_tables), to_dev(lens), c.B, int(lens.max()), d))
    torch.cuda.synchronize()
    assert_out_close(to_host(out), c.decode_ref(), "noalloc decode, peaked scores")
    st, flags = hyb.hyb_device_status(clear=True)
    assert st == 0, f"device status {flags:#x}"


def test_noalloc_decode_rejects_batches_beyond_its_scratch(hyb):
    H, D, B, msl = 32, 128, 64, 1 << 16               # partials need > 16 MiB
    d = hyb.dims(H, D, 10, msl // 16, W.BF16)
    assert hyb.hyb_paged_attn_decode_workspace_size(B, msl, d) > 16 << 20
    f = 1 << 20                                        # never dereferenced: rejected first
    assert hyb.hyb_paged_attn_decode_noalloc(f, f, f, f + 4096, f, f, B, msl, d) == hyb.HYB_ERR_UNSUPPORTED
