"""GPU parity at the named workload shapes: the tiny fp32 hybrid pair end to end, the
32-request single-layer decode batch at full size, the 32-layer hybrid decode through
the dispatcher, and the 8 x 131072-token long-context decode (sampled)."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import (lin_ws, as_f64, assert_out_close, assert_states_close, empty_rows,
                         poisoned_pool, same_bytes, to_dev, to_host)
from test_gpu_decode import DecodeStep

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------------ tiny pair
def _tiny_flow(hyb, use_dispatch, chunk):
    """Prefill prompts 5 and 37 through one Full and one Linear layer, then 4 decode steps.
    Returns every GPU result (host arrays) and the oracle's."""
    cfg = W.tiny_hybrid_pair(0)
    H, D, g, pool = cfg["H"], cfg["D"], cfg["g"], cfg["pool"]
    prompts, steps = cfg["prompts"], cfg["steps"]
    B, NB, MB = 2, pool.num_blocks, pool.max_blocks
    scale = 1 / math.sqrt(D)
    d = hyb.dims(H, D, NB, MB, W.F32, scale)
    cu = W.cu_from_lens(prompts)
    T = int(cu[-1])
    full_in = [W.rows(g, (T, H, D), D, W.F32) for _ in range(3)]
    lin_in = [W.rows(g, (T, H, D), D, W.F32) for _ in range(3)]
    dec_full = [[W.rows(g, (B, H, D), D, W.F32) for _ in range(3)] for _ in range(steps)]
    dec_lin = [[W.rows(g, (B, H, D), D, W.F32) for _ in range(3)] for _ in range(steps)]
    junk = W.synthetic_state(g, 3, H, D, np.array([50, 60, 70]))    # a previous request's leftovers
    slots = np.array([2, 0], np.int32)
    reset = np.array([1, 1], np.uint8)

    # ---- GPU
    bt = to_dev(pool.block_tables)
    kc = to_dev(poisoned_pool(NB, H, D, W.F32))
    vc = to_dev(poisoned_pool(NB, H, D, W.F32))
    st_pool = to_dev(junk)
    res = {"full_out": [], "lin_out": [], "slots": []}
    slot = torch.empty(T, dtype=torch.int64, device="cuda")
    hyb.check(hyb.hyb_slot_mapping(slot, bt, to_dev(cu), None, B, T, d))
    res["slots"].append(to_host(slot))
    fo = torch.empty((T, H, D), device="cuda")
    lo = torch.empty((T, H, D), device="cuda")
    q, k, v = (to_dev(a) for a in full_in)
    ql, kl, vl = (to_dev(a) for a in lin_in)
    cu_d, slots_d, reset_d = to_dev(cu), to_dev(slots), to_dev(reset)
    if use_dispatch:
        meta = hyb.batch_meta(B, T, block_tables=bt, slot_mapping=slot, cu_q_lens=cu_d,
                              state_slots=slots_d, reset=reset_d, max_q_len=int(prompts.max()))
        layers = [hyb.layer_io(fo, q, k, v, kc, vc), hyb.layer_io(lo, ql, kl, vl, state_pool=st_pool, num_state_slots=3)]
        hyb.check(hyb.hyb_layer_dispatch([0, 1], 2, 1, layers, meta, d, chunk, *lin_ws()))
    else:
        hyb.check(hyb.hyb_paged_kv_append(k, v, slot, T, kc, vc, d))
        hyb.check(hyb.hyb_paged_attn_prefill_causal(fo, q, kc, vc, bt, cu_d, None, B, T, int(prompts.max()), d))
        hyb.check(hyb.hyb_linear_attn_chunked_prefill(lo, ql, kl, vl, cu_d, None, st_pool, 3, slots_d,
                                                      reset_d, B, T, int(prompts.max()), H, D, chunk, W.F32, *lin_ws()))
    res["full_out"].append(to_host(fo))
    res["lin_out"].append(to_host(lo))
    ws = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    for s in range(steps):
        lens = prompts + s + 1
        lens_d = to_dev(lens.astype(np.int32))
        ctx_d = to_dev((lens - 1).astype(np.int32))
        slot = torch.empty(B, dtype=torch.int64, device="cuda")
        hyb.check(hyb.hyb_slot_mapping(slot, bt, to_dev(np.arange(B + 1, dtype=np.int32)), ctx_d, B, B, d))
        res["slots"].append(to_host(slot))
        q, k, v = (to_dev(a) for a in dec_full[s])
        ql, kl, vl = (to_dev(a) for a in dec_lin[s])
        fo = torch.empty((B, H, D), device="cuda")
        lo = torch.empty((B, H, D), device="cuda")
        if use_dispatch:
            meta = hyb.batch_meta(B, B, seq_lens=lens_d, block_tables=bt, slot_mapping=slot,
                                  state_slots=slots_d, max_seq_len=int(lens.max()))
            layers = [hyb.layer_io(fo, q, k, v, kc, vc), hyb.layer_io(lo, ql, kl, vl, state_pool=st_pool, num_state_slots=3)]
            hyb.check(hyb.hyb_layer_dispatch([0, 1], 2, 0, layers, meta, d, chunk, ws, 1 << 16))
        else:
            hyb.check(hyb.hyb_paged_kv_append(k, v, slot, B, kc, vc, d))
            hyb.check(hyb.hyb_paged_attn_decode(fo, q, kc, vc, bt, lens_d, B, int(lens.max()), d, ws, 1 << 16))
            hyb.check(hyb.hyb_linear_attn_step(lo, ql, kl, vl, st_pool, 3, slots_d, B, H, D, W.F32))
        res["full_out"].append(to_host(fo))
        res["lin_out"].append(to_host(lo))
    torch.cuda.synchronize()
    res["kc"], res["vc"], res["state"] = to_host(kc), to_host(vc), to_host(st_pool)

    # ---- oracle, on its own copies
    ref = {"full_out": [], "slots": []}
    okc, ovc = poisoned_pool(NB, H, D, W.F32), poisoned_pool(NB, H, D, W.F32)
    sm = oracle.slot_mapping(pool.block_tables, cu)
    ref["slots"].append(sm)
    oracle.kv_append(full_in[1], full_in[2], sm, okc, ovc)
    ref["full_out"].append(oracle.full_prefill(full_in[0], okc, ovc, pool.block_tables, cu, None, scale))
    for s in range(steps):
        lens = prompts + s + 1
        sm = oracle.slot_mapping(pool.block_tables, np.arange(B + 1), lens - 1)
        ref["slots"].append(sm)
        oracle.kv_append(dec_full[s][1], dec_full[s][2], sm, okc, ovc)
        ref["full_out"].append(oracle.full_decode(dec_full[s][0], okc, ovc, pool.block_tables, lens, scale))
    ref["kc"], ref["vc"] = okc, ovc
    # the linear layer's whole history per request, as one recurrence from the reset
    per_req = []
    for b in range(B):
        rows = [np.concatenate([lin_in[i][cu[b]:cu[b + 1]]] + [dec_lin[s][i][b:b + 1] for s in range(steps)])
                for i in range(3)]
        o, st = oracle.linear_recurrence(rows[0], rows[1], rows[2], [0, len(rows[0])])
        per_req.append((o, st[0]))
    ref["lin_prefill"] = np.concatenate([per_req[b][0][:prompts[b]] for b in range(B)])
    ref["lin_decode"] = [np.stack([per_req[b][0][prompts[b] + s] for b in range(B)]) for s in range(steps)]
    ref["state"] = np.stack([per_req[b][1] for b in range(B)])
    return res, ref, slots, junk


@pytest.mark.parametrize("chunk", [64, 1, 4, 16])
def test_tiny_hybrid_pair_matches_oracle(hyb, devstatus, chunk):
    res, ref, slots, junk = _tiny_flow(hyb, use_dispatch=False, chunk=chunk)
    for a, b in zip(res["slots"], ref["slots"]):
        assert np.array_equal(a, b)
    assert np.array_equal(res["kc"].view(np.uint32), ref["kc"].view(np.uint32))
    assert np.array_equal(res["vc"].view(np.uint32), ref["vc"].view(np.uint32))
    for a, b in zip(res["full_out"], ref["full_out"]):
        assert_out_close(a, b, "full")
    assert_out_close(res["lin_out"][0], ref["lin_prefill"], "linear prefill")
    for s in range(4):
        assert_out_close(res["lin_out"][s + 1], ref["lin_decode"][s], "linear decode")
    assert_states_close(res["state"][slots], ref["state"])
    assert np.array_equal(res["state"][1], junk[1])      # the slot nobody uses is untouched
    assert devstatus() == (0, 0)


def test_tiny_hybrid_pair_dispatch_equals_per_op_calls(hyb, devstatus):
    a, _, _, _ = _tiny_flow(hyb, use_dispatch=False, chunk=64)
    b, _, _, _ = _tiny_flow(hyb, use_dispatch=True, chunk=64)
    for key in ("full_out", "lin_out", "slots"):
        for x, y in zip(a[key], b[key]):
            assert np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8)), key
    for key in ("kc", "vc", "state"):
        assert np.array_equal(a[key].view(np.uint32), b[key].view(np.uint32)), key
    assert devstatus() == (0, 0)


# ------------------------------------------------------- 32-request decode batch
def test_single_layer_decode_batch_full_size(hyb, devstatus):
    """32 requests, H=32, D=128, seq_lens ~ U{128..4096}: every output against the oracle."""
    db = W.decode_single_layer(0)
    case = DecodeStep(0, db.seq_lens, db.H, db.D, db.dtype, pool=db.pool)
    sm_ref, kc_ref, vc_ref, out_ref = case.oracle_run()
    slot, kc, vc, out = case.gpu_run(hyb)
    assert np.array_equal(to_host(slot), sm_ref)
    # every appended row landed bit-exactly (the rest of the image is checked on small cases)
    kh = to_host(kc)
    for b, s in enumerate(sm_ref):
        assert np.array_equal(kh[s // 16, :, s % 16], case.k[b])
    del kh
    assert_out_close(out, out_ref, "decode out")
    # the bench's launch: the append fused into the decode, slots from the block table;
    # bit-identical to the separate append + decode above
    d = case.dims(hyb)
    msl = int(db.seq_lens.max())
    ws_n = hyb.hyb_paged_attn_decode_workspace_size(db.B, msl, d)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device="cuda")
    kc2, vc2 = to_dev(case.kc), to_dev(case.vc)
    out2 = empty_rows((db.B, db.H, db.D), db.dtype)
    hyb.check(hyb.hyb_paged_attn_decode_append(out2, to_dev(case.q), to_dev(case.k), to_dev(case.v), None, kc2, vc2,
                                               to_dev(db.pool.block_tables), to_dev(db.seq_lens), db.B, msl, d,
                                               ws, ws_n))
    torch.cuda.synchronize()
    assert torch.equal(out2.view(torch.int16), out.view(torch.int16))
    assert torch.equal(kc2.view(torch.int16), kc.view(torch.int16))
    assert torch.equal(vc2.view(torch.int16), vc.view(torch.int16))
    del kc2, vc2
    # Linear step at the same shape (state 32 x 128 x 128 fp32 per request)
    g = W.rng(1)
    B, H, D = db.B, db.H, db.D
    pool = W.synthetic_state(g, B, H, D, db.seq_lens)
    slots = g.permutation(B).astype(np.int32)
    q, k, v = (W.rows(g, (B, H, D), D, W.BF16) for _ in range(3))
    o_ref, s_ref = oracle.linear_step(q, k, v, pool, slots)
    pool_d = to_dev(pool)
    o = empty_rows((B, H, D), W.BF16)
    hyb.check(hyb.hyb_linear_attn_step(o, to_dev(q), to_dev(k), to_dev(v), pool_d, B, to_dev(slots), B, H, D, W.BF16))
    assert_out_close(o, o_ref, "linear out")
    assert_states_close(to_host(pool_d)[slots], s_ref)
    assert devstatus() == (0, 0)


# ------------------------------------------------------------- long context
@pytest.mark.parametrize("fused", [False, True])
def test_long_context_decode_sampled(hyb, devstatus, fused):
    """8 requests x 131072 tokens (8192 blocks each, randomly placed): sampled (request,
    head) pairs against the oracle, appended rows bit-exact, Linear step in full. `fused`:
    the append runs inside the decode (slots from the block table), as the bench's step."""
    db = W.decode_long_context(0)
    B, H, D, NB = db.B, db.H, db.D, db.pool.num_blocks
    n = int(db.seq_lens[0])
    kc = torch.empty((NB, H, 16, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.empty_like(kc)
    W.device_rows_(kc, 11, D)
    W.device_rows_(vc, 12, D)
    g = W.rng(5)
    q, k, v = (W.rows(g, (B, H, D), D, W.BF16) for _ in range(3))
    bt = db.pool.block_tables
    pairs = [(0, 0), (3, 17), (5, 31), (7, 8)]
    # oracle inputs gathered from the seeded pool BEFORE the GPU writes anything
    gathered = {}
    for b, h in pairs:
        blocks = torch.from_numpy(bt[b, :n // 16].astype(np.int64)).cuda()
        gathered[(b, h)] = (to_host(kc[blocks, h].reshape(n // 16, 1, 16, D)),
                            to_host(vc[blocks, h].reshape(n // 16, 1, 16, D)))
    d = hyb.dims(H, D, NB, db.pool.max_blocks, W.BF16)
    slot = torch.empty(B, dtype=torch.int64, device="cuda")
    out = empty_rows((B, H, D), W.BF16)
    ws_n = hyb.hyb_paged_attn_decode_workspace_size(B, n, d)
    ws = torch.empty(ws_n, dtype=torch.uint8, device="cuda")
    lens_d = to_dev(db.seq_lens)
    sm_ref = oracle.slot_mapping(bt, np.arange(B + 1), db.seq_lens - 1)
    if fused:
        hyb.check(hyb.hyb_paged_attn_decode_append(out, to_dev(q), to_dev(k), to_dev(v), None, kc, vc,
                                                   to_dev(bt), lens_d, B, n, d, ws, ws_n))
        torch.cuda.synchronize()
        sm = sm_ref
    else:
        hyb.check(hyb.hyb_slot_mapping(slot, to_dev(bt), to_dev(np.arange(B + 1, dtype=np.int32)),
                                       to_dev(db.seq_lens - 1), B, B, d))
        hyb.check(hyb.hyb_paged_kv_append(to_dev(k), to_dev(v), slot, B, kc, vc, d))
        hyb.check(hyb.hyb_paged_attn_decode(out, to_dev(q), kc, vc, to_dev(bt), lens_d, B, n, d, ws, ws_n))
        torch.cuda.synchronize()
        sm = to_host(slot)
        assert np.array_equal(sm, sm_ref)
    for b in range(B):
        s = int(sm[b])
        assert np.array_equal(to_host(kc[s // 16, :, s % 16]), k[b])
        assert np.array_equal(to_host(vc[s // 16, :, s % 16]), v[b])
    outh = to_host(out)
    for (b, h), (kg, vg) in gathered.items():
        ident = np.arange(n // 16, dtype=np.int32)[None, :]
        oracle.kv_append(k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1], np.array([n - 1], np.int64), kg, vg)
        ref = oracle.full_decode(q[b:b + 1, h:h + 1], kg, vg, ident, [n], 1 / math.sqrt(D))
        assert_out_close(outh[b:b + 1, h:h + 1], ref, f"decode ({b},{h})")
    del kc, vc
    # Linear step, 8 requests x 32 heads x 128 x 128 fp32
    pool = W.synthetic_state(g, B, H, D, db.seq_lens)
    slots = np.arange(B, dtype=np.int32)[::-1].copy()
    ql, kl, vl = (W.rows(g, (B, H, D), D, W.BF16) for _ in range(3))
    o_ref, s_ref = oracle.linear_step(ql, kl, vl, pool, slots)
    pool_d = to_dev(pool)
    o = empty_rows((B, H, D), W.BF16)
    hyb.check(hyb.hyb_linear_attn_step(o, to_dev(ql), to_dev(kl), to_dev(vl), pool_d, B, to_dev(slots), B, H, D, W.BF16))
    assert_out_close(o, o_ref)
    assert_states_close(to_host(pool_d)[slots], s_ref)
    assert devstatus() == (0, 0)


# ---------------------------------------------------- 32-layer hybrid decode
@pytest.mark.parametrize("slot_from_table", [False, True])
def test_hybrid_32_layer_dispatch(hyb, devstatus, slot_from_table):
    """layer_types = [F,F,F,Lin] x 8, batch 64 with the 80/20 short/long mix: the dispatcher
    equals per-op calls bit for bit (outputs, caches, states), and layers 0 (Full) and 3
    (Linear) match the oracle. `slot_from_table`: no slot mapping in the metadata, so each
    Full layer finds the new row's slot through the block table (the bench's 32-layer step)."""
    db = W.decode_hybrid_32layer(0)
    lt = db.extra["layer_types"]
    B, H, D, NB, MB = db.B, db.H, db.D, db.pool.num_blocks, db.pool.max_blocks
    d = hyb.dims(H, D, NB, MB, W.BF16)
    g = W.rng(3)
    msl = int(db.seq_lens.max())
    bt, lens = to_dev(db.pool.block_tables), to_dev(db.seq_lens)
    slots = to_dev(g.permutation(B).astype(np.int32))
    layers_dev, host_in = [], []
    for l, t in enumerate(lt):
        q, k, v = (W.rows(g, (B, H, D), D, W.BF16) for _ in range(3))
        host_in.append((q, k, v))
        io = dict(out=empty_rows((B, H, D), W.BF16), q=to_dev(q), k=to_dev(k), v=to_dev(v))
        if t == 0:
            io["k_cache"] = W.device_rows_(torch.empty((NB, H, 16, D), dtype=torch.bfloat16, device="cuda"), 1000 + l, D)
            io["v_cache"] = W.device_rows_(torch.empty((NB, H, 16, D), dtype=torch.bfloat16, device="cuda"), 2000 + l, D)
        else:
            io["state_pool"] = W.device_state_(torch.empty((B, H, D, D), device="cuda"), 3000 + l, db.seq_lens, D)
        layers_dev.append(io)
    before = {0: (to_host(layers_dev[0]["k_cache"]), to_host(layers_dev[0]["v_cache"])),
              3: to_host(layers_dev[3]["state_pool"]),
              30: (to_host(layers_dev[30]["k_cache"]), to_host(layers_dev[30]["v_cache"])),
              31: to_host(layers_dev[31]["state_pool"])}
    clones = [{k2: (v2.clone() if k2 in ("k_cache", "v_cache", "state_pool") else v2) for k2, v2 in io.items()}
              for io in layers_dev]
    for io in clones:
        io["out"] = torch.empty_like(io["out"])
    slot = torch.empty(B, dtype=torch.int64, device="cuda")
    hyb.check(hyb.hyb_slot_mapping(slot, bt, to_dev(np.arange(B + 1, dtype=np.int32)),
                                   to_dev(db.seq_lens - 1), B, B, d))
    ws_n = hyb.hyb_paged_attn_decode_workspace_size(B, msl, d)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device="cuda")
    meta = hyb.batch_meta(B, B, seq_lens=lens, block_tables=bt, slot_mapping=None if slot_from_table else slot,
                          state_slots=slots, max_seq_len=msl)
    ios = [hyb.layer_io(io["out"], io["q"], io["k"], io["v"], io.get("k_cache"), io.get("v_cache"),
                        io.get("state_pool"), B) for io in layers_dev]
    hyb.check(hyb.hyb_layer_dispatch(lt, 32, 0, ios, meta, d, 64, ws, ws_n))
    for t, io in zip(lt, clones):      # the same plan, one op at a time
        if t == 0:
            hyb.check(hyb.hyb_paged_kv_append(io["k"], io["v"], slot, B, io["k_cache"], io["v_cache"], d))
            hyb.check(hyb.hyb_paged_attn_decode(io["out"], io["q"], io["k_cache"], io["v_cache"], bt, lens, B, msl, d, ws, ws_n))
        else:
            hyb.check(hyb.hyb_linear_attn_step(io["out"], io["q"], io["k"], io["v"], io["state_pool"], B, slots, B, H, D, W.BF16))
    torch.cuda.synchronize()
    for a, b in zip(layers_dev, clones):
        for key in ("out", "k_cache", "v_cache", "state_pool"):
            if key in a:
                assert torch.equal(a[key].view(torch.uint8) if a[key].dtype != torch.float32 else a[key].view(torch.int32),
                                   b[key].view(torch.uint8) if b[key].dtype != torch.float32 else b[key].view(torch.int32)), key
    # oracle on layer 0 (Full) and layer 3 (Linear), from the pre-dispatch copies
    kc0, vc0 = before[0]
    q, k, v = host_in[0]
    sm = oracle.slot_mapping(db.pool.block_tables, np.arange(B + 1), db.seq_lens - 1)
    assert np.array_equal(to_host(slot), sm)
    oracle.kv_append(k, v, sm, kc0, vc0)
    ref = oracle.full_decode(q, kc0, vc0, db.pool.block_tables, db.seq_lens, 1 / math.sqrt(D))
    assert_out_close(layers_dev[0]["out"], ref, "layer 0")
    del kc0, vc0
    q, k, v = host_in[3]
    o_ref, s_ref = oracle.linear_step(q, k, v, before[3], to_host(slots))
    assert_out_close(layers_dev[3]["out"], o_ref, "layer 3")
    assert_states_close(to_host(layers_dev[3]["state_pool"])[to_host(slots)], s_ref)
    # and the last Full and Linear layers, which read their cache / state before waiting
    # for the layer before them
    kc30, vc30 = before[30]
    q, k, v = host_in[30]
    oracle.kv_append(k, v, sm, kc30, vc30)
    ref = oracle.full_decode(q, kc30, vc30, db.pool.block_tables, db.seq_lens, 1 / math.sqrt(D))
    assert_out_close(layers_dev[30]["out"], ref, "layer 30")
    assert same_bytes(to_host(layers_dev[30]["k_cache"]), kc30) and same_bytes(to_host(layers_dev[30]["v_cache"]), vc30)
    del kc30, vc30
    q, k, v = host_in[31]
    o_ref, s_ref = oracle.linear_step(q, k, v, before[31], to_host(slots))
    assert_out_close(layers_dev[31]["out"], o_ref, "layer 31")
    assert_states_close(to_host(layers_dev[31]["state_pool"])[to_host(slots)], s_ref)
    assert devstatus() == (0, 0)


# ------------------------------------------------------- lifecycle / isolation
def test_checkpoint_resume_is_bit_identical(hyb):
    """Copy a request's state and KV to the host after one step, reload them into fresh
    buffers and keep decoding: identical to the uninterrupted run."""
    H, D, B = 4, 128, 2
    case = DecodeStep(21, [100, 300], H, D, W.BF16)
    g = W.rng(22)
    steps = [[W.rows(g, (B, H, D), D, W.BF16) for _ in range(3)] for _ in range(3)]
    d = case.dims(hyb)
    bt = to_dev(case.pool.block_tables)

    def run(kc, vc, st, s0, s1):
        outs = []
        for s in range(s0, s1):
            lens = case.lens + s
            q, k, v = (to_dev(a) for a in steps[s])
            slot = torch.empty(B, dtype=torch.int64, device="cuda")
            hyb.check(hyb.hyb_slot_mapping(slot, bt, to_dev(np.arange(B + 1, dtype=np.int32)), to_dev(lens - 1), B, B, d))
            hyb.check(hyb.hyb_paged_kv_append(k, v, slot, B, kc, vc, d))
            o = empty_rows((B, H, D), W.BF16)
            ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
            hyb.check(hyb.hyb_paged_attn_decode(o, q, kc, vc, bt, to_dev(lens), B, int(lens.max()), d, ws, 1 << 20))
            ol = empty_rows((B, H, D), W.BF16)
            hyb.check(hyb.hyb_linear_attn_step(ol, q, k, v, st, B, to_dev(np.arange(B, dtype=np.int32)), B, H, D, W.BF16))
            outs.append((to_host(o), to_host(ol)))
        return outs

    st0 = W.synthetic_state(g, B, H, D, case.lens)
    kc, vc, st = to_dev(case.kc), to_dev(case.vc), to_dev(st0)
    full = run(kc, vc, st, 0, 3)
    kc, vc, st = to_dev(case.kc), to_dev(case.vc), to_dev(st0)
    first = run(kc, vc, st, 0, 1)
    saved = (to_host(kc), to_host(vc), to_host(st))          # checkpoint on the host
    del kc, vc, st
    kc, vc, st = (to_dev(a) for a in saved)                  # resume in fresh buffers
    rest = run(kc, vc, st, 1, 3)
    for a, b in zip(full, first + rest):
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_dispatch_layers_use_only_their_own_pools(hyb, devstatus):
    """Canary pools that no layer owns stay byte-identical; each layer's pool changes only
    where its own op writes."""
    H, D, B = 2, 64, 3
    case = DecodeStep(31, [20, 33, 70], H, D, W.BF16)
    d = case.dims(hyb)
    g = W.rng(32)
    canary = torch.full((case.pool.num_blocks, H, 16, D), 3.0, dtype=torch.bfloat16, device="cuda")
    canary_state = torch.full((B, H, D, D), -2.0, device="cuda")
    layers, ios = [], []
    for l, t in enumerate([0, 1, 0]):
        q, k, v = (to_dev(W.rows(g, (B, H, D), D, W.BF16)) for _ in range(3))
        io = dict(out=empty_rows((B, H, D), W.BF16), q=q, k=k, v=v)
        if t == 0:
            io["k_cache"], io["v_cache"] = to_dev(case.kc), to_dev(case.vc)
        else:
            io["state_pool"] = torch.zeros((B, H, D, D), device="cuda")
        layers.append(io)
        ios.append(hyb.layer_io(io["out"], q, k, v, io.get("k_cache"), io.get("v_cache"), io.get("state_pool"), B))
    slot = torch.empty(B, dtype=torch.int64, device="cuda")
    hyb.check(hyb.hyb_slot_mapping(slot, to_dev(case.pool.block_tables), to_dev(case.cu), to_dev(case.ctx), B, B, d))
    meta = hyb.batch_meta(B, B, seq_lens=to_dev(case.lens), block_tables=to_dev(case.pool.block_tables),
                          slot_mapping=slot, state_slots=to_dev(np.arange(B, dtype=np.int32)), max_seq_len=70)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    hyb.check(hyb.hyb_layer_dispatch([0, 1, 0], 3, 0, ios, meta, d, 64, ws, 1 << 20))
    torch.cuda.synchronize()
    assert bool((canary.float() == 3.0).all()) and bool((canary_state == -2.0).all())
    sm = to_host(slot)
    for l in (0, 2):
        kh = to_host(layers[l]["k_cache"])
        diff = np.argwhere((kh != case.kc).any(axis=(1, 3)))      # (block, offset) pairs written
        written = sorted(int(b) * 16 + int(o) for b, o in diff)
        assert written == sorted(sm.tolist())
        for b in range(B):
            s = int(sm[b])
            assert np.array_equal(kh[s // 16, :, s % 16], to_host(layers[l]["k"])[b])
    assert devstatus() == (0, 0)


def test_dispatch_step_captured_in_cuda_graph_replays_bit_identically(hyb, devstatus):
    """A whole decode step (slot mapping + 4-layer dispatch) captured into a CUDA graph and
    replayed gives the same bytes as the eager calls (no allocation or synchronisation
    inside the step; first-call set-up happens before capture)."""
    H, D, B = 4, 128, 3
    lt = [0, 0, 1, 0]
    case = DecodeStep(41, [200, 33, 700], H, D, W.BF16)
    d = case.dims(hyb)
    g = W.rng(42)
    bt, lens = to_dev(case.pool.block_tables), to_dev(case.lens)
    cu, ctx = to_dev(case.cu), to_dev(case.ctx)
    slots = to_dev(np.arange(B, dtype=np.int32))
    ins = [[to_dev(W.rows(g, (B, H, D), D, W.BF16)) for _ in range(3)] for _ in lt]
    st0 = W.synthetic_state(g, B, H, D, case.lens)

    def make_state():
        caches = [(to_dev(case.kc), to_dev(case.vc)) if t == 0 else None for t in lt]
        pools = [to_dev(st0) if t == 1 else None for t in lt]
        outs = [empty_rows((B, H, D), W.BF16) for _ in lt]
        ios = [hyb.layer_io(outs[l], *ins[l], *(caches[l] or (None, None)), pools[l], B) for l in range(len(lt))]
        return caches, pools, outs, ios

    slot = torch.empty(B, dtype=torch.int64, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    meta = hyb.batch_meta(B, B, seq_lens=lens, block_tables=bt, slot_mapping=slot, state_slots=slots, max_seq_len=700)
    s = torch.cuda.Stream()

    def step(ios):
        hyb.check(hyb.hyb_slot_mapping(slot, bt, cu, ctx, B, B, d, s))
        hyb.check(hyb.hyb_layer_dispatch(lt, len(lt), 0, ios, meta, d, 64, ws, 1 << 20, s))

    eager = make_state()
    with torch.cuda.stream(s):
        step(eager[3])
    s.synchronize()
    graphed = make_state()
    warm = make_state()
    with torch.cuda.stream(s):
        step(warm[3])                            # first-call set-up outside the capture
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step(graphed[3])
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager[2], graphed[2]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    for a, b in zip(eager[0] + eager[1], graphed[0] + graphed[1]):
        if a is None:
            continue
        for x, y in (zip(a, b) if isinstance(a, tuple) else [(a, b)]):
            assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))
    assert devstatus() == (0, 0)


def test_dispatch_sees_inputs_written_just_before_it(hyb, devstatus):
    """Every layer of a decode dispatch after the first reads its lengths, block ids and cache
    tiles (a Linear layer: its state) before waiting for the kernel launched before it. Here
    every input of the call (q/k/v, caches, states and the batch metadata) is written on the
    same stream right before the dispatch, with no synchronisation, the largest copies last;
    the outputs, caches and states must equal per-op calls made after everything settled."""
    lens = np.array([3000, 40, 700, 5, 1500, 128, 513, 2048], np.int32)
    B, H, D = len(lens), 4, 128
    lt = [0, 0, 1, 0, 0, 0, 1, 0]
    g = W.rng(901)
    pool = W.block_pool(g, lens, slack=8.0)              # a big pool: long copies
    NB, MB = pool.num_blocks, pool.max_blocks
    d = hyb.dims(H, D, NB, MB, W.BF16)
    msl = int(lens.max())
    slots_h = g.permutation(B).astype(np.int32)
    true = []
    for l, t in enumerate(lt):
        x = {n: to_dev(W.rows(g, (B, H, D), D, W.BF16)) for n in ("q", "k", "v")}
        if t == 0:
            x["k_cache"] = W.device_rows_(torch.empty((NB, H, 16, D), dtype=torch.bfloat16, device="cuda"), 5000 + l, D)
            x["v_cache"] = W.device_rows_(torch.empty((NB, H, 16, D), dtype=torch.bfloat16, device="cuda"), 6000 + l, D)
        else:
            x["state_pool"] = W.device_state_(torch.empty((B, H, D, D), device="cuda"), 7000 + l, lens, D)
        true.append(x)
    meta_true = {"lens": to_dev(lens), "bt": to_dev(pool.block_tables), "slots": to_dev(slots_h)}
    torch.cuda.synchronize()
    # the dispatch's own buffers hold NaN / garbage until the copies below land
    bufs = [{n: torch.full_like(v, float("nan")) for n, v in x.items()} for x in true]
    outs = [torch.empty((B, H, D), dtype=torch.bfloat16, device="cuda") for _ in lt]
    meta_bufs = {"lens": torch.zeros_like(meta_true["lens"]), "bt": torch.full_like(meta_true["bt"], -1),
                 "slots": torch.full_like(meta_true["slots"], -1)}
    ws_n = hyb.hyb_paged_attn_decode_workspace_size(B, msl, d)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device="cuda")
    meta = hyb.batch_meta(B, B, seq_lens=meta_bufs["lens"], block_tables=meta_bufs["bt"],
                          state_slots=meta_bufs["slots"], max_seq_len=msl)
    ios = [hyb.layer_io(outs[l], b["q"], b["k"], b["v"], b.get("k_cache"), b.get("v_cache"), b.get("state_pool"), B)
           for l, b in enumerate(bufs)]
    s = torch.cuda.current_stream()
    for n in meta_bufs:
        meta_bufs[n].copy_(meta_true[n])
    for b, x in zip(bufs, true):
        for n in ("q", "k", "v"):
            b[n].copy_(x[n])
    for b, x in reversed(list(zip(bufs, true))):         # caches of the last layers last
        for n in ("k_cache", "v_cache", "state_pool"):
            if n in b:
                b[n].copy_(x[n])
    hyb.check(hyb.hyb_layer_dispatch(lt, len(lt), 0, ios, meta, d, 64, ws, ws_n, s.cuda_stream))
    torch.cuda.synchronize()
    # per-op reference on the settled inputs
    ref_out = []
    slot = torch.empty(B, dtype=torch.int64, device="cuda")
    hyb.check(hyb.hyb_slot_mapping(slot, meta_true["bt"], to_dev(np.arange(B + 1, dtype=np.int32)),
                                   to_dev(lens - 1), B, B, d))
    for t, x in zip(lt, true):
        o = torch.empty((B, H, D), dtype=torch.bfloat16, device="cuda")
        if t == 0:
            hyb.check(hyb.hyb_paged_kv_append(x["k"], x["v"], slot, B, x["k_cache"], x["v_cache"], d))
            hyb.check(hyb.hyb_paged_attn_decode(o, x["q"], x["k_cache"], x["v_cache"], meta_true["bt"],
                                                meta_true["lens"], B, msl, d, ws, ws_n))
        else:
            hyb.check(hyb.hyb_linear_attn_step(o, x["q"], x["k"], x["v"], x["state_pool"], B, meta_true["slots"],
                                               B, H, D, W.BF16))
        ref_out.append(o)
    torch.cuda.synchronize()
    for l, (b, x) in enumerate(zip(bufs, true)):
        assert torch.equal(outs[l].view(torch.int16), ref_out[l].view(torch.int16)), f"layer {l} output"
        for n in ("k_cache", "v_cache"):
            if n in b:
                assert torch.equal(b[n].view(torch.int16), x[n].view(torch.int16)), f"layer {l} {n}"
        if "state_pool" in b:
            assert torch.equal(b["state_pool"].view(torch.int32), x["state_pool"].view(torch.int32)), f"layer {l} state"
    assert devstatus() == (0, 0)
