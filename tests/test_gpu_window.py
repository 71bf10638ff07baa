"""GPU parity of sliding-window Full attention through the C ABI (a query at position i sees
keys i - W < p <= i): paged decode, tensor-core and CUDA-core prefill, and SLIDING layers in
the dispatch, against the CPU oracle. Blocks that end before a request's window may be
released (block-table entry -1): the kernels must neither read nor flag them."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import (lin_ws, PagedCase as Case, assert_out_close, decode_case as _decode_case,
                         decode_gpu as _decode_gpu, empty_rows, released as _released,
                         same_bytes, to_dev, to_host)

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------------------ decode
@pytest.mark.parametrize("dtype,H,D", [(W.BF16, 8, 128), (W.F32, 4, 64)])
@pytest.mark.parametrize("window", [1, 16, 17, 100, 512, 1000, 5000])
def test_window_decode_matches_oracle(hyb, devstatus, dtype, H, D, window):
    lens = [1, 15, 16, 17, 100, 513, 2000, 4096]
    c = _decode_case(300 + window, lens, H, D, dtype)
    ref = oracle.full_decode(c.q, c.okc, c.ovc, c.pool.block_tables, c.ctx + 1, c.scale, window=window)
    out, ws_n = _decode_gpu(hyb, c, window, c.pool.block_tables)
    assert_out_close(out, ref, f"decode W={window}")
    # released blocks before each window: never read, never flagged, same bytes out
    out_r, _ = _decode_gpu(hyb, c, window, _released(c.pool.block_tables, c.ctx, window))
    assert same_bytes(to_host(out_r), to_host(out))
    assert devstatus() == (0, 0)
    # the workspace shrinks with the window (no split covers blocks outside it)
    d_full = c.dims(hyb, 0)
    assert ws_n <= hyb.hyb_paged_attn_decode_workspace_size(c.B, int(c.ctx.max()) + 1, d_full)


def test_window_covering_sequence_equals_full_decode_bit_exact(hyb, devstatus):
    c = _decode_case(310, [3, 700, 4096], 8, 128, W.BF16)
    full, _ = _decode_gpu(hyb, c, 0, c.pool.block_tables)
    win, _ = _decode_gpu(hyb, c, 4096, c.pool.block_tables)
    assert same_bytes(to_host(win), to_host(full))
    assert devstatus() == (0, 0)


def test_window_decode_single_layer_workload(hyb, devstatus):
    """32 requests, lengths 128..4096, H=32, D=128, window 1024: every output element."""
    db = W.decode_single_layer(0)
    lens = db.seq_lens
    c = _decode_case(320, lens, db.H, db.D, W.BF16)
    ref = oracle.full_decode(c.q, c.okc, c.ovc, c.pool.block_tables, lens, c.scale, window=1024)
    out, _ = _decode_gpu(hyb, c, 1024, _released(c.pool.block_tables, c.ctx, 1024))
    assert_out_close(out, ref, "decode W=1024")
    assert devstatus() == (0, 0)


# ----------------------------------------------------------------------- prefill
@pytest.mark.parametrize("window", [1, 16, 100, 128, 129, 1000])
@pytest.mark.parametrize("qlens,ctx", [
    ([1, 5, 127, 128, 129, 300], [0] * 6),
    ([77, 256, 1, 130], [16, 300, 511, 5]),
])
def test_window_prefill_tensor_core_matches_oracle(hyb, devstatus, window, qlens, ctx):
    c = Case(400 + window + len(qlens), qlens, ctx, 4, 128, W.BF16)
    ref = c.prefill_ref(window)
    out, slot, kc = c.prefill_gpu(hyb, window, c.pool.block_tables)
    assert np.array_equal(slot, c.sm) and same_bytes(kc, c.okc)
    assert_out_close(out, ref, f"prefill W={window}")
    out_r, *_ = c.prefill_gpu(hyb, window, _released(c.pool.block_tables, c.ctx, window))
    assert same_bytes(to_host(out_r), to_host(out))
    assert devstatus() == (0, 0)


@pytest.mark.parametrize("window", [0, 1, 200])
def test_cuda_core_prefill_long_context_matches_oracle(hyb, devstatus, window):
    """fp32, D=64 (no tensor-core kernel): contexts past 512 keys, with and without window."""
    c = Case(450 + window, [40, 3, 600], [700, 1030, 0], 4, 64, W.F32)
    ref = c.prefill_ref(window)
    bt = c.pool.block_tables if window == 0 else _released(c.pool.block_tables, c.ctx, window)
    out, slot, kc = c.prefill_gpu(hyb, window, bt)
    assert np.array_equal(slot, c.sm)
    assert_out_close(out, ref, f"cuda-core prefill W={window}")
    assert devstatus() == (0, 0)


def test_window_prefill_full_workload_sampled(hyb, devstatus):
    """8 requests x 8192 tokens, H=32, D=128, window 4096 (tensor-core kernel); sampled rows
    on both sides of the window edge against the oracle."""
    pb = W.prefill_chunked(0)
    B, H, D, NB = len(pb.q_lens), pb.H, pb.D, pb.pool.num_blocks
    cu = W.cu_from_lens(pb.q_lens)
    T = int(cu[-1])
    g = W.rng(460)
    q, k, v = (W.rows(g, (T, H, D), D, W.BF16) for _ in range(3))
    scale = 1 / math.sqrt(D)
    d = hyb.dims(H, D, NB, pb.pool.max_blocks, W.BF16, scale, window=4096)
    kc = torch.zeros((NB, H, 16, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    bt, cu_d = to_dev(pb.pool.block_tables), to_dev(cu)
    slot = torch.empty(T, dtype=torch.int64, device="cuda")
    hyb.check(hyb.hyb_slot_mapping(slot, bt, cu_d, None, B, T, d))
    hyb.check(hyb.hyb_paged_kv_append(to_dev(k), to_dev(v), slot, T, kc, vc, d))
    out = empty_rows((T, H, D), W.BF16)
    hyb.check(hyb.hyb_paged_attn_prefill_causal(out, to_dev(q), kc, vc, bt, cu_d, None, B, T, 8192, d))
    torch.cuda.synchronize()
    sm = oracle.slot_mapping(pb.pool.block_tables, cu)
    rng = np.random.default_rng(5)
    rows = sorted(set([int(cu[b]) + j for b in range(B) for j in (0, 4095, 4096, 4097, 8191)] +
                      rng.integers(0, T, 16).tolist()))
    okc = np.zeros((NB, H, 16, D), np.uint16)
    ovc = okc.copy()
    oracle.kv_append(k, v, sm, okc, ovc)
    ref = oracle.full_prefill(q, okc, ovc, pb.pool.block_tables, cu, None, scale, window=4096,
                              rows=np.array(rows, np.int32))
    assert_out_close(to_host(out)[rows], ref, "windowed prefill rows")
    assert devstatus() == (0, 0)


# ---------------------------------------------------------------------- dispatch
@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("mode", [0, 1])
def test_dispatch_sliding_layers_equal_per_op_calls(hyb, devstatus, mode, bs):
    """Layers FULL, SLIDING(64), LINEAR, SLIDING(700), 16- and 32-token blocks: the dispatch
    equals the per-op calls bit for bit, and the windowed layers match the oracle."""
    H, D = 4, 128
    types = [hyb.HYB_FULL, hyb.HYB_SLIDING, hyb.HYB_LINEAR, hyb.HYB_SLIDING]
    windows = [0, 64, 0, 700]
    if mode == 0:
        c = _decode_case(470, [1, 65, 900, 2000], H, D, W.BF16, bs)
    else:
        c = Case(471, [100, 700, 33], [0, 64, 1024], H, D, W.BF16, bs)   # Linear: chunk-aligned starts
    B, T = c.B, c.T
    d0 = c.dims(hyb, 0)                                   # carries the block size
    bt, cu_d, ctx_d = to_dev(c.pool.block_tables), to_dev(c.cu), to_dev(c.ctx)
    lens_d = to_dev(c.ctx + c.qlens)
    slot = torch.empty(T, dtype=torch.int64, device="cuda")
    hyb.check(hyb.hyb_slot_mapping(slot, bt, cu_d, ctx_d, B, T, d0))
    msl = int((c.ctx + c.qlens).max())
    # one workspace for both modes: decode partials, or the Linear prefill's handoff flags
    ws_n = max(hyb.hyb_paged_attn_decode_workspace_size(B, msl, d0), hyb.hyb_linear_attn_chunked_prefill_workspace_size())
    ws = torch.empty(ws_n, dtype=torch.uint8, device="cuda")
    st0 = W.synthetic_state(W.rng(472), B, H, D, c.ctx + c.qlens)
    slots_d = to_dev(np.arange(B, dtype=np.int32))
    reset_d = to_dev(np.zeros(B, np.uint8))
    q, k, v = to_dev(c.q), to_dev(c.k), to_dev(c.v)

    def fresh():
        return ([to_dev(c.kc) if t != hyb.HYB_LINEAR else None for t in types],
                [to_dev(c.vc) if t != hyb.HYB_LINEAR else None for t in types],
                [to_dev(st0) if t == hyb.HYB_LINEAR else None for t in types],
                [empty_rows((T, H, D), W.BF16) for _ in types])

    # dispatch
    kcs, vcs, pools, outs = fresh()
    ios = [hyb.layer_io(outs[l], q, k, v, kcs[l], vcs[l], pools[l], B if pools[l] is not None else 0,
                        window=windows[l]) for l in range(4)]
    meta = hyb.batch_meta(B, T, seq_lens=lens_d, block_tables=bt, slot_mapping=slot, cu_q_lens=cu_d,
                          ctx_lens=ctx_d, state_slots=slots_d, reset=reset_d, max_seq_len=msl,
                          max_q_len=int(c.qlens.max()))
    hyb.check(hyb.hyb_layer_dispatch(types, 4, mode, ios, meta, d0, 64, ws, ws_n))
    # per-op calls
    kcs2, vcs2, pools2, outs2 = fresh()
    for l, t in enumerate(types):
        if t == hyb.HYB_LINEAR:
            if mode == 0:
                hyb.check(hyb.hyb_linear_attn_step(outs2[l], q, k, v, pools2[l], B, slots_d, B, H, D, W.BF16))
            else:
                hyb.check(hyb.hyb_linear_attn_chunked_prefill(outs2[l], q, k, v, cu_d, ctx_d, pools2[l], B,
                                                              slots_d, reset_d, B, T, int(c.qlens.max()),
                                                              H, D, 64, W.BF16, *lin_ws()))
            continue
        dl = c.dims(hyb, windows[l])
        hyb.check(hyb.hyb_paged_kv_append(k, v, slot, T, kcs2[l], vcs2[l], dl))
        if mode == 0:
            hyb.check(hyb.hyb_paged_attn_decode(outs2[l], q, kcs2[l], vcs2[l], bt, lens_d, B, msl, dl, ws, ws_n))
        else:
            hyb.check(hyb.hyb_paged_attn_prefill_causal(outs2[l], q, kcs2[l], vcs2[l], bt, cu_d, ctx_d, B, T,
                                                        int(c.qlens.max()), dl))
    torch.cuda.synchronize()
    for l in range(4):
        assert same_bytes(to_host(outs[l]), to_host(outs2[l])), f"layer {l}"
    for l in (1, 3):
        ref = c.decode_ref(windows[l]) if mode == 0 else c.prefill_ref(windows[l])
        assert_out_close(outs[l], ref, f"sliding layer {l}")
    assert devstatus() == (0, 0)
