"""GPU parity of the tensor-core prefill paths through the C ABI: causal prefill over the
paged cache (incl. a cached prefix) and chunked linear prefill (state carried across
chunks and calls), against the CPU oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import (lin_ws, assert_out_close, assert_states_close, empty_rows, poisoned_pool,
                         same_bytes, to_dev, to_host)

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------ causal prefill
def _prefill_case(hyb, seed, qlens, ctx, H=4, D=128):
    g = W.rng(seed)
    qlens = np.asarray(qlens, np.int32)
    ctx = np.asarray(ctx, np.int32)
    tot = qlens + ctx
    pool = W.block_pool(g, tot)
    # the cached prefix (ctx rows per request), written by the oracle into a poisoned pool
    cu_ctx = W.cu_from_lens(ctx)
    kp, vp = (W.rows(g, (int(cu_ctx[-1]), H, D), D, W.BF16) for _ in range(2))
    kc = poisoned_pool(pool.num_blocks, H, D, W.BF16)
    vc = kc.copy()
    oracle.kv_append(kp, vp, oracle.slot_mapping(pool.block_tables, cu_ctx), kc, vc)
    cu = W.cu_from_lens(qlens)
    T = int(cu[-1])
    q, k, v = (W.rows(g, (T, H, D), D, W.BF16) for _ in range(3))
    scale = 1 / math.sqrt(D)
    # oracle: append this call's rows, then causal attention
    sm = oracle.slot_mapping(pool.block_tables, cu, ctx)
    okc, ovc = kc.copy(), vc.copy()
    oracle.kv_append(k, v, sm, okc, ovc)
    ref = oracle.full_prefill(q, okc, ovc, pool.block_tables, cu, ctx, scale)
    # GPU
    d = hyb.dims(H, D, pool.num_blocks, pool.max_blocks, W.BF16, scale)
    bt, cu_d, ctx_d = to_dev(pool.block_tables), to_dev(cu), to_dev(ctx)
    kcd, vcd = to_dev(kc), to_dev(vc)
    slot = torch.empty(T, dtype=torch.int64, device="cuda")
    hyb.check(hyb.hyb_slot_mapping(slot, bt, cu_d, ctx_d, len(qlens), T, d))
    hyb.check(hyb.hyb_paged_kv_append(to_dev(k), to_dev(v), slot, T, kcd, vcd, d))
    out = empty_rows((T, H, D), W.BF16)
    hyb.check(hyb.hyb_paged_attn_prefill_causal(out, to_dev(q), kcd, vcd, bt, cu_d, ctx_d, len(qlens), T,
                                                int(qlens.max()), d))
    torch.cuda.synchronize()
    return out, ref, (to_host(slot), sm), (to_host(kcd), okc)


@pytest.mark.parametrize("qlens,ctx", [
    ([1, 5, 127, 128, 129, 300], [0] * 6),
    ([1000, 64, 200], [0, 0, 0]),
    ([77, 256, 1, 130], [16, 300, 511, 5]),          # chunked prefill over a cached prefix
])
def test_causal_prefill_tensor_core_matches_oracle(hyb, devstatus, qlens, ctx):
    out, ref, (s_gpu, s_ref), (kc_gpu, kc_ref) = _prefill_case(hyb, 50 + len(qlens), qlens, ctx)
    assert np.array_equal(s_gpu, s_ref)
    assert same_bytes(kc_gpu, kc_ref)
    assert_out_close(out, ref, "prefill")
    assert devstatus() == (0, 0)


def test_prefill_rows_equal_decode_of_same_prefix(hyb, devstatus):
    """The last row of a prefill equals a decode step over the same cached prefix."""
    out, ref, *_ = _prefill_case(hyb, 61, [300, 129], [0, 40])
    assert_out_close(out[[299, 428]], ref[[299, 428]])
    assert devstatus() == (0, 0)


@pytest.mark.parametrize("B,L", [(8, 8192), (2, 32768)])
def test_causal_prefill_full_workload_sampled(hyb, devstatus, B, L):
    """8 requests x 8192 tokens (and 2 x 32768, the longest prompts the prefill-length bench
    row runs), H=32, D=128: KV appended to a shuffled pool, tensor-core causal prefill;
    sampled rows (incl. first/last of every request) against the oracle."""
    pb = W.prefill_chunked(0, B=B, L=L)
    B, H, D, NB = len(pb.q_lens), pb.H, pb.D, pb.pool.num_blocks
    cu = W.cu_from_lens(pb.q_lens)
    T = int(cu[-1])
    g = W.rng(71)
    q, k, v = (W.rows(g, (T, H, D), D, W.BF16) for _ in range(3))
    scale = 1 / math.sqrt(D)
    d = hyb.dims(H, D, NB, pb.pool.max_blocks, W.BF16, scale)
    kc = torch.zeros((NB, H, 16, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    bt, cu_d = to_dev(pb.pool.block_tables), to_dev(cu)
    slot = torch.empty(T, dtype=torch.int64, device="cuda")
    hyb.check(hyb.hyb_slot_mapping(slot, bt, cu_d, None, B, T, d))
    hyb.check(hyb.hyb_paged_kv_append(to_dev(k), to_dev(v), slot, T, kc, vc, d))
    out = empty_rows((T, H, D), W.BF16)
    hyb.check(hyb.hyb_paged_attn_prefill_causal(out, to_dev(q), kc, vc, bt, cu_d, None, B, T, L, d))
    torch.cuda.synchronize()
    sm = oracle.slot_mapping(pb.pool.block_tables, cu)
    assert np.array_equal(to_host(slot), sm)
    rng = np.random.default_rng(3)
    rows = sorted(set([int(cu[b]) for b in range(B)] + [int(cu[b + 1]) - 1 for b in range(B)] +
                      [int(cu[b]) + j for b in range(B) for j in (127, 128, 4095, L - 129)] +
                      rng.integers(0, T, 24).tolist()))
    # oracle cache image built by the oracle itself (same bytes as the inputs)
    okc = np.zeros((NB, H, 16, D), np.uint16)
    ovc = okc.copy()
    oracle.kv_append(k, v, sm, okc, ovc)
    ref = oracle.full_prefill(q, okc, ovc, pb.pool.block_tables, cu, None, scale, rows=np.array(rows, np.int32))
    assert_out_close(to_host(out)[rows], ref, "prefill rows")
    assert devstatus() == (0, 0)


# ------------------------------------------------------- chunked linear prefill
def _linear_case(seed, lens, H=4, D=128, NS=None, with_state=True):
    g = W.rng(seed)
    lens = np.asarray(lens, np.int32)
    B = len(lens)
    NS = NS or B + 2
    cu = W.cu_from_lens(lens)
    T = int(cu[-1])
    q, k, v = (W.rows(g, (T, H, D), D, W.BF16) for _ in range(3))
    pool = W.synthetic_state(g, NS, H, D, np.full(NS, 500)) if with_state else np.zeros((NS, H, D, D), np.float32)
    slots = g.permutation(NS)[:B].astype(np.int32)
    reset = (g.integers(0, 2, B)).astype(np.uint8)
    return dict(q=q, k=k, v=v, cu=cu, T=T, pool=pool, slots=slots, reset=reset, B=B, H=H, D=D, NS=NS, lens=lens)


def _linear_gpu(hyb, c, chunk=64, ctx=None, pool_d=None):
    pool_d = to_dev(c["pool"]) if pool_d is None else pool_d
    out = empty_rows((c["T"], c["H"], c["D"]), W.BF16)
    hyb.check(hyb.hyb_linear_attn_chunked_prefill(
        out, to_dev(c["q"]), to_dev(c["k"]), to_dev(c["v"]), to_dev(c["cu"]),
        None if ctx is None else to_dev(np.asarray(ctx, np.int32)), pool_d, c["NS"], to_dev(c["slots"]),
        to_dev(c["reset"]), c["B"], c["T"], int(c["lens"].max()), c["H"], c["D"], chunk, W.BF16, *lin_ws()))
    torch.cuda.synchronize()
    return out, pool_d


@pytest.mark.parametrize("lens", [[1, 63, 64, 65, 130, 300], [1000, 7, 640]])
def test_chunked_linear_tensor_core_matches_recurrence(hyb, devstatus, lens):
    c = _linear_case(80 + len(lens), lens)
    o_ref, s_ref = oracle.linear_recurrence(c["q"], c["k"], c["v"], c["cu"], c["pool"], c["slots"], c["reset"])
    out, pool_d = _linear_gpu(hyb, c)
    assert_out_close(out, o_ref, "linear prefill out")
    got = to_host(pool_d)
    assert_states_close(got[c["slots"]], s_ref, "linear prefill state")
    untouched = np.setdiff1d(np.arange(c["NS"]), c["slots"])
    assert np.array_equal(got[untouched], c["pool"][untouched])
    assert devstatus() == (0, 0)


def test_chunked_linear_split_calls_equal_one_call(hyb, devstatus):
    """A prompt prefilled in two calls split at a chunk boundary (state carried in the
    pool) equals one call, and both equal the recurrence."""
    H, D, n, split = 4, 128, 700, 384
    g = W.rng(90)
    q, k, v = (W.rows(g, (n, H, D), D, W.BF16) for _ in range(3))
    o_ref, s_ref = oracle.linear_recurrence(q, k, v, [0, n])
    pool = torch.zeros((1, H, D, D), device="cuda")
    outs = []
    lws = lin_ws()                                       # one workspace, calls in stream order
    for lo, hi in ((0, split), (split, n)):
        out = empty_rows((hi - lo, H, D), W.BF16)
        hyb.check(hyb.hyb_linear_attn_chunked_prefill(
            out, to_dev(q[lo:hi]), to_dev(k[lo:hi]), to_dev(v[lo:hi]), to_dev(np.array([0, hi - lo], np.int32)),
            to_dev(np.array([lo], np.int32)), pool, 1, to_dev(np.zeros(1, np.int32)),
            to_dev(np.array([1 if lo == 0 else 0], np.uint8)), 1, hi - lo, hi - lo, H, D, 64, W.BF16, *lws))
        outs.append(to_host(out))
    torch.cuda.synchronize()
    assert_out_close(np.concatenate(outs), o_ref)
    assert_states_close(to_host(pool), s_ref)
    assert devstatus() == (0, 0)


def test_chunked_linear_misaligned_start_is_flagged(hyb, devstatus):
    c = _linear_case(91, [100, 50], H=2)
    before = c["pool"].copy()
    out, pool_d = _linear_gpu(hyb, c, ctx=[64, 10])              # request 1 starts mid-chunk
    st, flags = devstatus()
    assert flags == hyb.HYB_DEVERR_MISALIGNED
    assert np.array_equal(to_host(pool_d)[c["slots"][1]], before[c["slots"][1]])   # left alone
    o_ref, s_ref = oracle.linear_recurrence(c["q"][:100], c["k"][:100], c["v"][:100], [0, 100], c["pool"],
                                            c["slots"][:1], c["reset"][:1])
    assert_out_close(out[:100], o_ref)


def test_chunked_linear_many_chains_ragged(hyb, devstatus):
    """More (request, head) chains than SMs with ragged lengths: empty requests (reset or
    not), one row, exactly one chunk, partial last chunks, one long request. Every output
    row and every state against the recurrence. The kernel shares all chunks out evenly
    over its CTAs, so here chains are cut between CTAs at many points and several short
    chains follow one another inside one CTA."""
    g = W.rng(95)
    lens = g.integers(0, 700, 48)
    lens[[3, 17, 30]] = 0
    lens[[5, 6, 7]] = [1, 64, 129]
    lens[40] = 2500
    c = _linear_case(96, lens, H=8)
    c["reset"][[3, 17]] = 1                              # an empty request with a reset: zero state
    c["reset"][30] = 0                                   # and one without: state left alone
    o_ref, s_ref = oracle.linear_recurrence(c["q"], c["k"], c["v"], c["cu"], c["pool"], c["slots"], c["reset"])
    out, pool_d = _linear_gpu(hyb, c)
    assert_out_close(out, o_ref, "linear prefill out")
    got = to_host(pool_d)
    assert_states_close(got[c["slots"]], s_ref, "linear prefill state")
    assert not got[c["slots"][[3, 17]]].any()
    assert np.array_equal(got[c["slots"][30]], c["pool"][c["slots"][30]])
    untouched = np.setdiff1d(np.arange(c["NS"]), c["slots"])
    assert np.array_equal(got[untouched], c["pool"][untouched])
    assert devstatus() == (0, 0)


def test_chunked_linear_graph_replays_with_new_inputs(hyb, devstatus):
    """The prefill captured once in a CUDA graph and replayed with new q/k/v and a fresh
    state each time: every replay equals the recurrence on its own inputs (so no replay
    takes a state handed over by an earlier one)."""
    c = _linear_case(97, np.full(40, 300), H=8)
    qd, kd, vd = (to_dev(c[x]) for x in ("q", "k", "v"))
    cu_d, slots_d, reset_d = to_dev(c["cu"]), to_dev(c["slots"]), to_dev(c["reset"])
    pool_d = to_dev(c["pool"])
    out = empty_rows((c["T"], c["H"], c["D"]), W.BF16)
    lws = lin_ws()                                       # kept for every replay

    def call():
        hyb.check(hyb.hyb_linear_attn_chunked_prefill(out, qd, kd, vd, cu_d, None, pool_d, c["NS"], slots_d,
                                                      reset_d, c["B"], c["T"], 300, c["H"], c["D"], 64, W.BF16, *lws))

    call()                                               # first call outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for rep in range(3):
        g = W.rng(300 + rep)
        new = {x: W.rows(g, (c["T"], c["H"], c["D"]), c["D"], W.BF16) for x in ("q", "k", "v")}
        for x, d in (("q", qd), ("k", kd), ("v", vd)):
            d.copy_(to_dev(new[x]))
        pool_d.copy_(to_dev(c["pool"]))
        graph.replay()
        torch.cuda.synchronize()
        o_ref, s_ref = oracle.linear_recurrence(new["q"], new["k"], new["v"], c["cu"], c["pool"], c["slots"],
                                                c["reset"])
        assert_out_close(out, o_ref, f"replay {rep}")
        assert_states_close(to_host(pool_d)[c["slots"]], s_ref, f"replay {rep} state")
    assert devstatus() == (0, 0)


def test_chunked_linear_two_streams_at_once(hyb, devstatus):
    """Two chunked-prefill calls, each with its own handoff workspace, issued on two streams
    back to back, four times: grids of 16 CTAs leave room for both to be resident at once,
    and the unequal chains (16 and 3 chunks) make each call hand states between its CTAs.
    Both calls finish without a handoff timeout and each equals the recurrence on its own
    inputs: a call only ever reads its own workspace's flags."""
    cases = [_linear_case(700 + i, [2000, 300], H=8) for i in range(2)]
    refs = [oracle.linear_recurrence(c["q"], c["k"], c["v"], c["cu"], c["pool"], c["slots"], c["reset"])
            for c in cases]
    dev = []
    for c in cases:
        dev.append(dict(q=to_dev(c["q"]), k=to_dev(c["k"]), v=to_dev(c["v"]), cu=to_dev(c["cu"]),
                        slots=to_dev(c["slots"]), reset=to_dev(c["reset"]), ws=lin_ws(),
                        out=empty_rows((c["T"], c["H"], c["D"]), W.BF16)))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for rep in range(4):
        pools = [to_dev(c["pool"]) for c in cases]
        torch.cuda.synchronize()
        for c, x, pool, s in zip(cases, dev, pools, streams):
            hyb.check(hyb.hyb_linear_attn_chunked_prefill(
                x["out"], x["q"], x["k"], x["v"], x["cu"], None, pool, c["NS"], x["slots"], x["reset"], c["B"],
                c["T"], int(c["lens"].max()), c["H"], c["D"], 64, W.BF16, *x["ws"], s))
        torch.cuda.synchronize()
        for i, (c, x, pool, (o_ref, s_ref)) in enumerate(zip(cases, dev, pools, refs)):
            assert_out_close(x["out"], o_ref, f"call {i}, round {rep}")
            assert_states_close(to_host(pool)[c["slots"]], s_ref, f"call {i}, round {rep} state")
        assert devstatus() == (0, 0)


def test_chunked_linear_full_workload_sampled(hyb, devstatus):
    """8 requests x 8192 tokens, H=32, D=128, chunk 64, zero initial state: whole output
    shape computed on the GPU; sampled (request, head) chains against the recurrence."""
    pb = W.prefill_chunked(0)
    B, H, D = len(pb.q_lens), pb.H, pb.D
    cu = W.cu_from_lens(pb.q_lens)
    T = int(cu[-1])
    g = W.rng(72)
    q, k, v = (W.rows(g, (T, H, D), D, W.BF16) for _ in range(3))
    pool = torch.full((B, H, D, D), 5.0, device="cuda")          # garbage: every request resets
    slots = np.arange(B, dtype=np.int32)
    out = empty_rows((T, H, D), W.BF16)
    hyb.check(hyb.hyb_linear_attn_chunked_prefill(out, to_dev(q), to_dev(k), to_dev(v), to_dev(cu), None, pool, B,
                                                  to_dev(slots), to_dev(np.ones(B, np.uint8)), B, T, 8192, H, D, 64,
                                                  W.BF16, *lin_ws()))
    torch.cuda.synchronize()
    outh, st = to_host(out), to_host(pool)
    for b, h in [(0, 0), (0, 1), (3, 17), (5, 9), (7, 31)]:
        sl = slice(int(cu[b]), int(cu[b + 1]))
        o_ref, s_ref = oracle.linear_recurrence(q[sl, h:h + 1], k[sl, h:h + 1], v[sl, h:h + 1], [0, 8192])
        assert_out_close(outh[sl, h:h + 1], o_ref, f"chain ({b},{h})")
        assert_states_close(st[b, h:h + 1], s_ref[0], f"state ({b},{h})")
    assert devstatus() == (0, 0)


def test_prefill_dispatch_equals_per_op_calls(hyb, devstatus):
    """hyb_layer_dispatch in prefill mode (Full: append + tensor-core causal prefill;
    Linear: tensor-core chunked prefill) equals the per-op calls bit for bit."""
    H, D = 4, 128
    lens = np.array([200, 64, 513], np.int32)
    B = len(lens)
    g = W.rng(95)
    pool = W.block_pool(g, lens)
    cu = W.cu_from_lens(lens)
    T = int(cu[-1])
    d = hyb.dims(H, D, pool.num_blocks, pool.max_blocks, W.BF16)
    ins = [[to_dev(W.rows(g, (T, H, D), D, W.BF16)) for _ in range(3)] for _ in range(2)]
    bt, cu_d = to_dev(pool.block_tables), to_dev(cu)
    slots, reset = to_dev(np.arange(B, dtype=np.int32)), to_dev(np.ones(B, np.uint8))
    res = []
    for use_dispatch in (False, True):
        kc = torch.zeros((pool.num_blocks, H, 16, D), dtype=torch.bfloat16, device="cuda")
        vc = torch.zeros_like(kc)
        st = torch.zeros((B, H, D, D), device="cuda")
        fo, lo = empty_rows((T, H, D), W.BF16), empty_rows((T, H, D), W.BF16)
        slot = torch.empty(T, dtype=torch.int64, device="cuda")
        hyb.check(hyb.hyb_slot_mapping(slot, bt, cu_d, None, B, T, d))
        (q, k, v), (ql, kl, vl) = ins
        if use_dispatch:
            meta = hyb.batch_meta(B, T, block_tables=bt, slot_mapping=slot, cu_q_lens=cu_d, state_slots=slots,
                                  reset=reset, max_q_len=int(lens.max()))
            hyb.check(hyb.hyb_layer_dispatch([0, 1], 2, 1, [hyb.layer_io(fo, q, k, v, kc, vc),
                                                            hyb.layer_io(lo, ql, kl, vl, state_pool=st, num_state_slots=B)],
                                             meta, d, 64, *lin_ws()))
        else:
            hyb.check(hyb.hyb_paged_kv_append(k, v, slot, T, kc, vc, d))
            hyb.check(hyb.hyb_paged_attn_prefill_causal(fo, q, kc, vc, bt, cu_d, None, B, T, int(lens.max()), d))
            hyb.check(hyb.hyb_linear_attn_chunked_prefill(lo, ql, kl, vl, cu_d, None, st, B, slots, reset, B, T,
                                                          int(lens.max()), H, D, 64, W.BF16, *lin_ws()))
        torch.cuda.synchronize()
        res.append([to_host(x) for x in (fo, lo, kc, vc, st)])
    for a, b in zip(*res):
        assert same_bytes(a, b)
    assert devstatus() == (0, 0)
