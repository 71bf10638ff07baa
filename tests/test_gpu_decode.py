"""GPU parity of the decode path through the C ABI: slot mapping, KV append, paged decode,
linear step -- against the CPU oracle on the same seeded bytes."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import (as_f64, assert_out_close, assert_states_close, empty_rows,
                         poisoned_pool, same_bytes, to_dev, to_host)

pytestmark = pytest.mark.gpu


class DecodeStep:
    """One decode token per request over a paged pool whose prefix (seq_len - 1 rows per
    request) was written by the oracle; q/k/v of the new token are fresh seeded rows."""

    def __init__(self, seed, lens, H, D, dtype, slack=1.25, pool=None):
        g = W.rng(seed)
        self.lens = np.asarray(lens, np.int32)
        self.B, self.H, self.D, self.dtype = len(self.lens), H, D, dtype
        self.pool = pool if pool is not None else W.block_pool(g, np.maximum(self.lens, 1), slack=slack)
        prev = np.maximum(self.lens - 1, 0)
        cu_prev = W.cu_from_lens(prev)
        kp = W.rows(g, (int(cu_prev[-1]), H, D), D, dtype)
        vp = W.rows(g, (int(cu_prev[-1]), H, D), D, dtype)
        self.kc = poisoned_pool(self.pool.num_blocks, H, D, dtype)
        self.vc = self.kc.copy()
        oracle.kv_append(kp, vp, oracle.slot_mapping(self.pool.block_tables, cu_prev), self.kc, self.vc)
        self.q, self.k, self.v = (W.rows(g, (self.B, H, D), D, dtype) for _ in range(3))
        self.scale = 1 / math.sqrt(D)
        self.cu = np.arange(self.B + 1, dtype=np.int32)
        self.ctx = np.maximum(self.lens - 1, 0).astype(np.int32)

    def oracle_run(self):
        sm = oracle.slot_mapping(self.pool.block_tables, self.cu, self.ctx)
        kc, vc = self.kc.copy(), self.vc.copy()
        oracle.kv_append(self.k, self.v, sm, kc, vc)
        out = oracle.full_decode(self.q, kc, vc, self.pool.block_tables, self.lens, self.scale)
        return sm, kc, vc, out

    def dims(self, hyb):
        return hyb.dims(self.H, self.D, self.pool.num_blocks, self.pool.max_blocks, self.dtype,
                        self.scale)

    def gpu_run(self, hyb, kc=None, vc=None, max_seq_len=None):
        d = self.dims(hyb)
        dev = dict(bt=to_dev(self.pool.block_tables), lens=to_dev(self.lens), cu=to_dev(self.cu),
                   ctx=to_dev(self.ctx), q=to_dev(self.q), k=to_dev(self.k), v=to_dev(self.v))
        kc = to_dev(self.kc) if kc is None else kc
        vc = to_dev(self.vc) if vc is None else vc
        slot = torch.empty(self.B, dtype=torch.int64, device="cuda")
        out = empty_rows((self.B, self.H, self.D), self.dtype)
        msl = int(self.lens.max()) if max_seq_len is None else max_seq_len
        ws_n = hyb.hyb_paged_attn_decode_workspace_size(self.B, msl, d)
        ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device="cuda")
        hyb.check(hyb.hyb_slot_mapping(slot, dev["bt"], dev["cu"], dev["ctx"], self.B, self.B, d))
        hyb.check(hyb.hyb_paged_kv_append(dev["k"], dev["v"], slot, self.B, kc, vc, d))
        hyb.check(hyb.hyb_paged_attn_decode(out, dev["q"], kc, vc, dev["bt"], dev["lens"], self.B,
                                            msl, d, ws, ws_n))
        torch.cuda.synchronize()
        return slot, kc, vc, out


@pytest.mark.parametrize("dtype,H,D,lens", [
    (W.BF16, 32, 128, [1, 15, 16, 17, 31, 33, 511, 512, 513, 4095, 4096]),
    (W.BF16, 4, 64, [1, 2, 100, 1000]),
    (W.BF16, 2, 16, [3, 16, 48, 700]),
    (W.BF16, 3, 256, [5, 600]),
    (W.F32, 2, 16, [9, 41]),
    (W.F32, 4, 128, [1, 17, 530]),
])
def test_decode_step_matches_oracle(hyb, devstatus, dtype, H, D, lens):
    case = DecodeStep(100 + len(lens), lens, H, D, dtype)
    sm_ref, kc_ref, vc_ref, out_ref = case.oracle_run()
    slot, kc, vc, out = case.gpu_run(hyb)
    assert np.array_equal(to_host(slot), sm_ref)                       # bit-exact indexing
    assert same_bytes(to_host(kc), kc_ref) and same_bytes(to_host(vc), vc_ref)
    assert_out_close(out, out_ref, "decode out")
    assert devstatus() == (0, 0)


def test_decode_at_the_largest_batch_the_grid_takes(hyb, devstatus):
    """65 535 rows, the most the decode grid holds (rows are its y dimension): short rows with
    one split and every 1000th row long enough for two, so both the split kernel and the
    combine run over the whole batch; the step matches the oracle (slots bit-exact)."""
    B = 65535
    g = W.rng(555)
    lens = g.integers(1, 41, size=B).astype(np.int32)
    lens[::1000] = 600
    case = DecodeStep(556, lens, 1, 16, W.F32)
    sm_ref, kc_ref, vc_ref, out_ref = case.oracle_run()
    slot, kc, vc, out = case.gpu_run(hyb)
    assert np.array_equal(to_host(slot), sm_ref)
    assert same_bytes(to_host(kc), kc_ref) and same_bytes(to_host(vc), vc_ref)
    assert_out_close(out, out_ref, "decode out, 65535 rows")
    assert devstatus() == (0, 0)


def test_decode_zero_length_gives_zeros(hyb, devstatus):
    case = DecodeStep(7, [5, 1, 40], 4, 128, W.BF16)
    d = case.dims(hyb)
    lens = np.array([4, 0, 39], np.int32)          # attend to the oracle-written prefix only
    out = torch.full((3, 4, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    hyb.check(hyb.hyb_paged_attn_decode(out, to_dev(case.q), to_dev(case.kc), to_dev(case.vc),
                                        to_dev(case.pool.block_tables), to_dev(lens), 3, 48, d,
                                        ws, 1 << 20))
    ref = oracle.full_decode(case.q, case.kc, case.vc, case.pool.block_tables, lens, case.scale)
    assert not to_host(out[1]).any()
    assert_out_close(out, ref)
    assert devstatus() == (0, 0)


def test_decode_deterministic_and_batch_invariant(hyb):
    """Two identical launches agree bit for bit; a request alone equals the same request
    inside a batch (split-K depends only on the request's own length)."""
    lens = [4096, 130, 2000, 17]
    case = DecodeStep(8, lens, 32, 128, W.BF16)
    _, kc, vc, out1 = case.gpu_run(hyb)
    d = case.dims(hyb)
    bt, ln, q = to_dev(case.pool.block_tables), to_dev(case.lens), to_dev(case.q)
    ws = torch.empty(1 << 24, dtype=torch.uint8, device="cuda")
    out2 = torch.empty_like(out1)
    hyb.check(hyb.hyb_paged_attn_decode(out2, q, kc, vc, bt, ln, 4, 4096, d, ws, 1 << 24))
    out3 = torch.empty_like(out1[2:3])
    hyb.check(hyb.hyb_paged_attn_decode(out3, q[2:3].contiguous(), kc, vc, bt[2:3].contiguous(),
                                        ln[2:3].contiguous(), 1, 2000, d, ws, 1 << 24))
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(out1[2:3].view(torch.int16), out3.view(torch.int16))


def test_bad_block_id_is_flagged_and_skipped(hyb, devstatus):
    case = DecodeStep(9, [40, 40], 2, 128, W.BF16)
    bt = case.pool.block_tables.copy()
    bt[1, 1] = case.pool.num_blocks + 5           # out of the pool: must not be read
    d = case.dims(hyb)
    out = empty_rows((2, 2, 128), W.BF16)
    ws = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    lens = np.array([39, 39], np.int32)           # the oracle-written prefix (no append here)
    hyb.check(hyb.hyb_paged_attn_decode(out, to_dev(case.q), to_dev(case.kc), to_dev(case.vc),
                                        to_dev(bt), to_dev(lens), 2, 40, d, ws, 1 << 16))
    st, flags = devstatus()
    assert st == hyb.HYB_ERR_DEVICE_CHECK and flags & hyb.HYB_DEVERR_BAD_BLOCK
    # request 0 is untouched by request 1's bad entry; prefix rows 0..38 exist (39 appended)
    ref = oracle.full_decode(case.q[:1], case.kc, case.vc, case.pool.block_tables[:1], [39], case.scale)
    assert_out_close(out[:1], ref)
    assert torch.isfinite(out.float()).all()


def test_slot_minus_one_and_out_of_pool_slot(hyb, devstatus):
    H, D = 2, 16
    d = hyb.dims(H, D, 4, 4, W.F32)
    k = to_dev(W.rows(W.rng(3), (3, H, D), D, W.F32))
    kc = torch.zeros((4, H, 16, D), device="cuda")
    vc = torch.zeros_like(kc)
    slot = to_dev(np.array([5, -1, 64], np.int64))   # 64 = 4 blocks x 16: beyond the pool
    hyb.check(hyb.hyb_paged_kv_append(k, k, slot, 3, kc, vc, d))
    st, flags = devstatus()
    assert flags == hyb.HYB_DEVERR_BAD_SLOT
    ref = np.zeros((4, H, 16, D), np.float32)
    oracle.kv_append(to_host(k)[:2], to_host(k)[:2], np.array([5, -1], np.int64), ref, ref.copy())
    assert np.array_equal(to_host(kc), ref)


# ----------------------------------------------------------------- linear step
@pytest.mark.parametrize("dtype,H,D,B", [(W.BF16, 32, 128, 16), (W.BF16, 4, 64, 3),
                                         (W.F32, 2, 16, 2), (W.BF16, 2, 256, 2),
                                         (W.F32, 3, 32, 5)])
def test_linear_step_matches_oracle(hyb, devstatus, dtype, H, D, B):
    g = W.rng(200 + D)
    NS = B + 3
    seq = g.integers(1, 4000, size=NS)
    pool = W.synthetic_state(g, NS, H, D, seq)
    slots = g.permutation(NS)[:B].astype(np.int32)
    q, k, v = (W.rows(g, (B, H, D), D, dtype) for _ in range(3))
    out_ref, st_ref = oracle.linear_step(q, k, v, pool, slots)
    pool_d = to_dev(pool)
    out = empty_rows((B, H, D), dtype)
    hyb.check(hyb.hyb_linear_attn_step(out, to_dev(q), to_dev(k), to_dev(v), pool_d, NS,
                                       to_dev(slots), B, H, D, dtype))
    got = to_host(pool_d)
    assert_out_close(out, out_ref, "linear out")
    assert_states_close(got[slots], st_ref, "linear state")
    untouched = np.setdiff1d(np.arange(NS), slots)
    assert np.array_equal(got[untouched], pool[untouched])          # other slots bit-identical
    assert devstatus() == (0, 0)


def test_linear_zero_state_one_token_is_exact_outer_product(hyb):
    """A zeroed state plus one token holds exactly k (outer) v (bf16 x bf16 is exact in fp32)."""
    H, D, B = 32, 128, 4
    g = W.rng(11)
    q, k, v = (W.rows(g, (B, H, D), D, W.BF16) for _ in range(3))
    pool = torch.zeros((B, H, D, D), device="cuda")
    out = empty_rows((B, H, D), W.BF16)
    hyb.check(hyb.hyb_linear_attn_step(out, to_dev(q), to_dev(k), to_dev(v), pool, B,
                                       to_dev(np.arange(B, dtype=np.int32)), B, H, D, W.BF16))
    _, st_ref = oracle.linear_step(q, k, v, np.zeros((B, H, D, D), np.float32), np.arange(B))
    assert np.array_equal(to_host(pool).astype(np.float64), st_ref)


def test_linear_bad_state_slot_flagged(hyb, devstatus):
    H, D = 2, 16
    g = W.rng(12)
    q, k, v = (W.rows(g, (2, H, D), D, W.F32) for _ in range(3))
    pool = torch.zeros((2, H, D, D), device="cuda")
    out = empty_rows((2, H, D), W.F32)
    hyb.check(hyb.hyb_linear_attn_step(out, to_dev(q), to_dev(k), to_dev(v), pool, 2,
                                       to_dev(np.array([0, 9], np.int32)), 2, H, D, W.F32))
    st, flags = devstatus()
    assert flags == hyb.HYB_DEVERR_BAD_STATE
    assert not to_host(pool)[1].any()


def test_linear_decode_does_not_rezero_and_carries(hyb):
    """Consecutive steps carry the state (no re-zeroing between decode steps)."""
    H, D, n = 2, 64, 5
    g = W.rng(13)
    q, k, v = (W.rows(g, (n, 1, H, D), D, W.BF16) for _ in range(3))
    pool = torch.zeros((1, H, D, D), device="cuda")
    outs = []
    for t in range(n):
        out = empty_rows((1, H, D), W.BF16)
        hyb.check(hyb.hyb_linear_attn_step(out, to_dev(q[t]), to_dev(k[t]), to_dev(v[t]), pool, 1,
                                           to_dev(np.zeros(1, np.int32)), 1, H, D, W.BF16))
        outs.append(as_f64(out)[0])
    ref, st = oracle.linear_recurrence(q[:, 0], k[:, 0], v[:, 0], [0, n])
    assert_out_close(np.stack(outs), ref)
    assert_states_close(to_host(pool), st)
