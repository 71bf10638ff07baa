"""The dispatch trace (HYB_TRACE), a seeded randomized sweep of the decode step over head
dims, block sizes, lengths at block boundaries and skipped slots, and determinism of the
two prefill kernels (two identical launches agree bit for bit)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import lin_ws, assert_out_close, decode_case, empty_rows, same_bytes, to_dev, to_host

pytestmark = pytest.mark.gpu


def _decode_dispatch(hyb, c, layer_types, ios, lens):
    msl = int(lens.max())
    d = c.dims(hyb)
    ws_n = hyb.hyb_paged_attn_decode_workspace_size(c.B, msl, d)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device="cuda")
    slot = to_dev(np.asarray(c.sm, np.int64))
    meta = hyb.batch_meta(c.B, c.B, seq_lens=to_dev(lens), block_tables=to_dev(c.pool.block_tables),
                          slot_mapping=slot, state_slots=to_dev(np.arange(c.B, dtype=np.int32)), max_seq_len=msl)
    hyb.check(hyb.hyb_layer_dispatch(layer_types, len(layer_types), 0, ios, meta, d, 64, ws, ws_n))
    torch.cuda.synchronize()


def test_dispatch_trace_names_kernels_and_times_layers(hyb, devstatus, capfd, monkeypatch):
    c = decode_case(800, [20, 700, 3000], 4, 128, W.BF16)
    lens = c.ctx + 1
    kc1, vc1, kc2, vc2 = (to_dev(c.kc) for _ in range(4))
    st = torch.zeros((c.B, c.H, c.D, c.D), device="cuda")
    q, k, v = to_dev(c.q), to_dev(c.k), to_dev(c.v)

    def run():
        outs = [empty_rows((c.B, c.H, c.D), c.dtype) for _ in range(3)]
        ios = [hyb.layer_io(outs[0], q, k, v, kc1, vc1), hyb.layer_io(outs[1], q, k, v, kc2, vc2),
               hyb.layer_io(outs[2], q, k, v, state_pool=st, num_state_slots=c.B)]
        _decode_dispatch(hyb, c, [0, 0, 1], ios, lens)
        return [to_host(o) for o in outs]

    monkeypatch.delenv("HYB_TRACE", raising=False)
    plain = run()
    monkeypatch.setenv("HYB_TRACE", "1")
    capfd.readouterr()
    traced = run()
    err = capfd.readouterr().err
    assert all(same_bytes(a, b) for a, b in zip(plain[:2], traced[:2]))   # tracing changes nothing
    assert "dispatch decode, 3 layers" in err
    assert err.count("paged_decode_kernel (KV append fused)") == 2 and "linear_step_kernel" in err
    s, ms = hyb.hyb_trace_layer_ms(3)
    assert s == hyb.HYB_OK and all(t > 0 for t in ms), ms
    assert hyb.hyb_trace_layer_ms(2)[0] == hyb.HYB_ERR_INVALID_ARG        # fewer slots than layers
    assert devstatus() == (0, 0)


def _sweep_cases():
    g = np.random.default_rng(2024)
    cases = []
    for i in range(10):
        D = int(g.choice([16, 32, 64, 128]))
        dtype = W.F32 if i % 4 == 3 else W.BF16
        bs = int(g.choice([16, 32]))
        B = int(g.integers(1, 6))
        edges = [1, bs - 1, bs, bs + 1, 32 * 16, 32 * 16 + 1, 2 * bs * 16 - 1]
        lens = [int(g.choice(edges)) if g.random() < 0.5 else int(g.integers(1, 1500)) for _ in range(B)]
        cases.append((i, int(g.integers(1, 6)), D, dtype, bs, lens, int(g.integers(0, B))))
    return cases


@pytest.mark.parametrize("i,H,D,dtype,bs,lens,skip", _sweep_cases())
def test_decode_append_random_sweep(hyb, devstatus, i, H, D, dtype, bs, lens, skip):
    """Random shapes (seeded): the fused decode step against the oracle; one request's slot
    is -1 (nothing appended, the attention reads the cache as it is)."""
    c = decode_case(900 + i, lens, H, D, dtype, block_size=bs)
    slot_h = np.asarray(c.sm, np.int64).copy()
    slot_h[skip] = -1
    kc_ref, vc_ref = c.kc.copy(), c.vc.copy()
    oracle.kv_append(c.k, c.v, slot_h, kc_ref, vc_ref, bs)
    ref = oracle.full_decode(c.q, kc_ref, vc_ref, c.pool.block_tables, c.ctx + 1, c.scale, block_size=bs)
    d = c.dims(hyb)
    lens_a = c.ctx + 1
    msl = int(lens_a.max())
    kcd, vcd = to_dev(c.kc), to_dev(c.vc)
    ws_n = hyb.hyb_paged_attn_decode_workspace_size(c.B, msl, d)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device="cuda")
    out = empty_rows((c.B, c.H, c.D), c.dtype)
    hyb.check(hyb.hyb_paged_attn_decode_append(out, to_dev(c.q), to_dev(c.k), to_dev(c.v), to_dev(slot_h), kcd,
                                               vcd, to_dev(c.pool.block_tables), to_dev(lens_a), c.B, msl, d, ws,
                                               ws_n))
    torch.cuda.synchronize()
    assert same_bytes(to_host(kcd), kc_ref) and same_bytes(to_host(vcd), vc_ref)
    # the skipped request's newest position holds poison (NaN): its output is NaN in the
    # oracle too, so compare the others
    keep = np.arange(c.B) != skip
    assert_out_close(to_host(out)[keep], ref[keep], "sweep decode")
    assert devstatus() == (0, 0)


def test_prefill_kernels_are_deterministic(hyb, devstatus):
    """Two identical launches of the tensor-core causal prefill and of the chunked linear
    prefill give the same bytes (fixed reduction orders, no atomics in the arithmetic)."""
    g = W.rng(950)
    H, D = 8, 128
    lens = np.array([300, 1000, 4200, 77], np.int32)
    cu = W.cu_from_lens(lens)
    T = int(cu[-1])
    q, k, v = (to_dev(W.rows(g, (T, H, D), D, W.BF16)) for _ in range(3))
    pool = W.block_pool(g, lens)
    kc = to_dev(W.rows(g, (pool.num_blocks, H, 16, D), D, W.BF16))
    vc = to_dev(W.rows(g, (pool.num_blocks, H, 16, D), D, W.BF16))
    d = hyb.dims(H, D, pool.num_blocks, pool.max_blocks, W.BF16)
    bt, cu_d = to_dev(pool.block_tables), to_dev(cu)
    res = []
    for _ in range(2):
        out = empty_rows((T, H, D), W.BF16)
        hyb.check(hyb.hyb_paged_attn_prefill_causal(out, q, kc, vc, bt, cu_d, None, len(lens), T, int(lens.max()), d))
        lo = empty_rows((T, H, D), W.BF16)
        st = torch.zeros((len(lens), H, D, D), device="cuda")
        hyb.check(hyb.hyb_linear_attn_chunked_prefill(lo, q, k, v, cu_d, None, st, len(lens),
                                                      to_dev(np.arange(len(lens), dtype=np.int32)), None,
                                                      len(lens), T, int(lens.max()), H, D, 64, W.BF16, *lin_ws()))
        torch.cuda.synchronize()
        res.append((to_host(out), to_host(lo), to_host(st)))
    assert all(same_bytes(a, b) for a, b in zip(res[0], res[1]))
    assert devstatus() == (0, 0)
