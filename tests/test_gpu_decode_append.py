"""The decode step with the KV append fused into the decode launch
(hyb_paged_attn_decode_append): against the CPU oracle, and bit for bit against the two
separate calls (append, then decode) on the same bytes -- outputs and cache images."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import assert_out_close, decode_case, empty_rows, same_bytes, to_dev, to_host

pytestmark = pytest.mark.gpu


def _slots(c):
    """Slots of each request's new row (position seq_len - 1), by the oracle."""
    return oracle.slot_mapping(c.pool.block_tables, np.arange(c.B + 1, dtype=np.int32), c.ctx, c.bs)


def _run(hyb, c, slot_h, fused, window=0):
    """One decode step on the GPU from the case's prefix cache; returns (out, k cache, v cache)."""
    d = c.dims(hyb, window)
    lens = c.ctx + 1
    msl = int(lens.max())
    kcd, vcd = to_dev(c.kc), to_dev(c.vc)
    slot = to_dev(np.asarray(slot_h, np.int64))
    q, k, v = to_dev(c.q), to_dev(c.k), to_dev(c.v)
    bt, ln = to_dev(c.pool.block_tables), to_dev(lens)
    ws_n = hyb.hyb_paged_attn_decode_workspace_size(c.B, msl, d)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device="cuda")
    out = empty_rows((c.B, c.H, c.D), c.dtype)
    if fused:
        hyb.check(hyb.hyb_paged_attn_decode_append(out, q, k, v, slot, kcd, vcd, bt, ln, c.B, msl, d, ws, ws_n))
    else:
        hyb.check(hyb.hyb_paged_kv_append(k, v, slot, c.B, kcd, vcd, d))
        hyb.check(hyb.hyb_paged_attn_decode(out, q, kcd, vcd, bt, ln, c.B, msl, d, ws, ws_n))
    torch.cuda.synchronize()
    return to_host(out), to_host(kcd), to_host(vcd)


@pytest.mark.parametrize("dtype,H,D,lens,bs,window", [
    (W.BF16, 32, 128, [1, 15, 16, 17, 512, 513, 1000, 4096], 16, 0),
    (W.BF16, 4, 64, [2, 100, 1025, 3000], 32, 0),
    (W.BF16, 4, 128, [1, 300, 2049, 5000], 16, 700),
    (W.F32, 2, 16, [9, 41, 600], 16, 0),
])
def test_decode_append_matches_oracle_and_two_calls(hyb, devstatus, dtype, H, D, lens, bs, window):
    c = decode_case(700 + len(lens) + bs, lens, H, D, dtype, block_size=bs)
    slot_h = _slots(c)
    out_f, kc_f, vc_f = _run(hyb, c, slot_h, True, window)
    out_s, kc_s, vc_s = _run(hyb, c, slot_h, False, window)
    assert same_bytes(out_f, out_s)                      # same arithmetic, same order
    assert same_bytes(kc_f, kc_s) and same_bytes(vc_f, vc_s)
    assert same_bytes(kc_f, c.okc) and same_bytes(vc_f, c.ovc)   # the oracle's cache image
    assert_out_close(out_f, c.decode_ref(window), "fused decode")
    assert devstatus() == (0, 0)


def test_decode_append_skipped_and_bad_slots(hyb, devstatus):
    """slot -1: nothing written, the attention reads the cache as it is (same as the two
    calls); a slot beyond the pool: flagged, nothing written."""
    c = decode_case(720, [40, 300, 77], 4, 128, W.BF16)
    slot_h = _slots(c).copy()
    slot_h[1] = -1
    out_f, kc_f, vc_f = _run(hyb, c, slot_h, True)
    out_s, kc_s, vc_s = _run(hyb, c, slot_h, False)
    assert same_bytes(out_f, out_s) and same_bytes(kc_f, kc_s) and same_bytes(vc_f, vc_s)
    assert devstatus() == (0, 0)
    slot_h[2] = c.pool.num_blocks * c.bs                 # one past the pool
    before_k = c.kc.copy()                               # bf16 bit patterns (uint16)
    out_f, kc_f, _ = _run(hyb, c, slot_h, True)
    st, flags = devstatus()
    assert flags == hyb.HYB_DEVERR_BAD_SLOT
    # rows 0 (written) and 2 (refused): only row 0's slot changed
    changed = np.argwhere(np.any(kc_f.view(np.uint16) != before_k.view(np.uint16), axis=-1))
    assert {(int(b), int(t)) for b, _, t in changed} == {(int(slot_h[0]) // c.bs, int(slot_h[0]) % c.bs)}


def test_dispatch_decode_uses_fused_append_bit_identically(hyb, devstatus):
    """The decode-mode dispatch (append fused) equals slot mapping + append + decode calls."""
    c = decode_case(730, [5, 130, 2000, 64], 8, 128, W.BF16)
    d = c.dims(hyb)
    lens = c.ctx + 1
    msl = int(lens.max())
    slot_h = _slots(c)
    out_s, kc_s, vc_s = _run(hyb, c, slot_h, False)
    kcd, vcd = to_dev(c.kc), to_dev(c.vc)
    slot = to_dev(np.asarray(slot_h, np.int64))
    ws_n = hyb.hyb_paged_attn_decode_workspace_size(c.B, msl, d)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device="cuda")
    out = empty_rows((c.B, c.H, c.D), c.dtype)
    q, k, v = to_dev(c.q), to_dev(c.k), to_dev(c.v)
    meta = hyb.batch_meta(c.B, c.B, seq_lens=to_dev(lens), block_tables=to_dev(c.pool.block_tables),
                          slot_mapping=slot, max_seq_len=msl)
    hyb.check(hyb.hyb_layer_dispatch([0], 1, 0, [hyb.layer_io(out, q, k, v, kcd, vcd)], meta, d, 64, ws, ws_n))
    torch.cuda.synchronize()
    assert same_bytes(to_host(out), out_s)
    assert same_bytes(to_host(kcd), kc_s) and same_bytes(to_host(vcd), vc_s)
    assert devstatus() == (0, 0)


def test_decode_append_without_slot_mapping(hyb, devstatus):
    """slot_mapping NULL: each new row goes to position seq_len - 1 through the block table,
    bit-identical to passing the slots hyb_slot_mapping computes; also through the dispatch."""
    c = decode_case(740, [1, 16, 17, 500, 2049], 4, 128, W.BF16, block_size=32)
    out_s, kc_s, vc_s = _run(hyb, c, _slots(c), True)
    d = c.dims(hyb)
    lens = c.ctx + 1
    msl = int(lens.max())
    ws_n = hyb.hyb_paged_attn_decode_workspace_size(c.B, msl, d)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device="cuda")
    q, k, v = to_dev(c.q), to_dev(c.k), to_dev(c.v)
    bt, ln = to_dev(c.pool.block_tables), to_dev(lens)
    for via_dispatch in (False, True):
        kcd, vcd = to_dev(c.kc), to_dev(c.vc)
        out = empty_rows((c.B, c.H, c.D), c.dtype)
        if via_dispatch:
            meta = hyb.batch_meta(c.B, c.B, seq_lens=ln, block_tables=bt, max_seq_len=msl)
            hyb.check(hyb.hyb_layer_dispatch([0], 1, 0, [hyb.layer_io(out, q, k, v, kcd, vcd)], meta, d, 64, ws, ws_n))
        else:
            hyb.check(hyb.hyb_paged_attn_decode_append(out, q, k, v, None, kcd, vcd, bt, ln, c.B, msl, d, ws, ws_n))
        torch.cuda.synchronize()
        assert same_bytes(to_host(out), out_s)
        assert same_bytes(to_host(kcd), kc_s) and same_bytes(to_host(vcd), vc_s)
    assert devstatus() == (0, 0)
