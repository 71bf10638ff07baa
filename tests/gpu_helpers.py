"""Shared helpers of the GPU parity tests: host <-> device copies of the seeded inputs,
and the tolerance rules the tests apply.

Tolerances (floating point): bf16/fp32 attention outputs pass when every element has
|gpu - ref| <= 2e-2 + 1e-2 * |ref| (the allclose reading of "2e-2 max-abs / 1e-2
relative"); fp32
linear states pass when, for every (request, head) matrix, max|gpu - ref| <=
1e-3 * max|ref|. Integer and byte results (slots, cache images) must be identical.
"""
import math

import numpy as np
import torch

import oracle
import workloads as W

OUT_ATOL = 2e-2
OUT_REL = 1e-2
STATE_REL = 1e-3


def to_dev(a: np.ndarray, dtype_code: int | None = None, device="cuda"):
    """numpy -> CUDA tensor. uint16 arrays are bf16 bit patterns."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def to_host(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def as_f64(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        a = to_host(a)
    return W.bf16_to_f32(a).astype(np.float64) if a.dtype == np.uint16 else a.astype(np.float64)


def empty_rows(shape, dtype_code, device="cuda"):
    return torch.empty(shape, dtype=torch.bfloat16 if dtype_code == W.BF16 else torch.float32,
                       device=device)


def assert_out_close(gpu, ref, what="output"):
    """Elementwise |gpu - ref| <= 2e-2 + 1e-2 * |ref| (allclose form of "2e-2 max-abs /
    1e-2 relative"), every value finite. Returns the max abs error."""
    g = as_f64(gpu)
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    if not g.size:
        return 0.0
    err = np.abs(g - ref)
    lim = OUT_ATOL + OUT_REL * np.abs(ref)
    worst = int(np.argmax(err - lim))
    assert (err <= lim).all(), (f"{what}: |err| {err.flat[worst]:.3e} > {lim.flat[worst]:.3e} "
                                f"at ref {ref.flat[worst]:.3e}; max abs err {err.max():.3e}")
    return float(err.max())


def same_bytes(a, b) -> bool:
    """Bitwise equality of two host arrays (NaN patterns included)."""
    a, b = np.ascontiguousarray(a), np.ascontiguousarray(b)
    return a.shape == b.shape and a.dtype == b.dtype and np.array_equal(a.view(np.uint8), b.view(np.uint8))


def assert_states_close(gpu, ref, what="state"):
    g = as_f64(gpu)
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    m = g.reshape(-1, g.shape[-2] * g.shape[-1])
    r = ref.reshape(-1, ref.shape[-2] * ref.shape[-1])
    err = np.abs(m - r).max(axis=1)
    lim = STATE_REL * np.abs(r).max(axis=1)
    bad = np.nonzero(err > np.maximum(lim, 0.0) + (lim == 0) * 0.0)[0]
    assert len(bad) == 0, f"{what}: {len(bad)} matrices off, worst rel {(err / np.maximum(np.abs(r).max(axis=1), 1e-30)).max():.3e}"
    return float((err / np.maximum(np.abs(r).max(axis=1), 1e-30)).max())


def poisoned_pool(num_blocks, H, D, dtype_code, block_size=W.BLOCK_SIZE):
    shape = (num_blocks, H, block_size, D)
    if dtype_code == W.BF16:
        return np.full(shape, 0x7FC0, np.uint16)
    return np.full(shape, np.nan, np.float32)


# ------------------------------------------------- paged requests with a cached prefix
def released(block_tables, first_pos, window, block_size=W.BLOCK_SIZE):
    """Copy of the table with -1 for every logical block that ends before the window of the
    request's earliest query (position first_pos[b])."""
    bt = block_tables.copy()
    for b, p in enumerate(first_pos):
        keep_from = max(0, int(p) - window + 1) // block_size
        bt[b, :keep_from] = -1
    return bt


class PagedCase:
    """Requests with a cached prefix (ctx rows, written by the oracle into a poisoned pool)
    and this call's q/k/v rows (qlens per request)."""

    def __init__(self, seed, qlens, ctx, H, D, dtype, block_size=W.BLOCK_SIZE):
        g = W.rng(seed)
        self.qlens = np.asarray(qlens, np.int32)
        self.ctx = np.asarray(ctx, np.int32)
        self.B, self.H, self.D, self.dtype = len(self.qlens), H, D, dtype
        self.bs = block_size
        self.pool = W.block_pool(g, self.qlens + self.ctx, block_size=block_size)
        cu_ctx = W.cu_from_lens(self.ctx)
        kp, vp = (W.rows(g, (int(cu_ctx[-1]), H, D), D, dtype) for _ in range(2))
        self.kc = poisoned_pool(self.pool.num_blocks, H, D, dtype, block_size)
        self.vc = self.kc.copy()
        oracle.kv_append(kp, vp, oracle.slot_mapping(self.pool.block_tables, cu_ctx, block_size=block_size),
                         self.kc, self.vc, block_size)
        self.cu = W.cu_from_lens(self.qlens)
        self.T = int(self.cu[-1])
        self.q, self.k, self.v = (W.rows(g, (self.T, H, D), D, dtype) for _ in range(3))
        self.scale = 1 / math.sqrt(D)
        self.sm = oracle.slot_mapping(self.pool.block_tables, self.cu, self.ctx, block_size)
        self.okc, self.ovc = self.kc.copy(), self.vc.copy()
        oracle.kv_append(self.k, self.v, self.sm, self.okc, self.ovc, block_size)

    def dims(self, hyb, window=0):
        return hyb.dims(self.H, self.D, self.pool.num_blocks, self.pool.max_blocks, self.dtype,
                        self.scale, block_size=self.bs, window=window)

    def prefill_ref(self, window=0):
        return oracle.full_prefill(self.q, self.okc, self.ovc, self.pool.block_tables, self.cu,
                                   self.ctx, self.scale, block_size=self.bs, window=window)

    def decode_ref(self, window=0):
        """Decode rows (one per request, qlens all 1) over the appended cache."""
        return oracle.full_decode(self.q, self.okc, self.ovc, self.pool.block_tables, self.ctx + 1,
                                  self.scale, block_size=self.bs, window=window)

    def prefill_gpu(self, hyb, window, bt):
        """Append with the full table, attend with `bt` (possibly with released blocks)."""
        d = self.dims(hyb, window)
        cu_d, ctx_d = to_dev(self.cu), to_dev(self.ctx)
        kcd, vcd = to_dev(self.kc), to_dev(self.vc)
        slot = torch.empty(self.T, dtype=torch.int64, device="cuda")
        hyb.check(hyb.hyb_slot_mapping(slot, to_dev(self.pool.block_tables), cu_d, ctx_d, self.B, self.T, d))
        hyb.check(hyb.hyb_paged_kv_append(to_dev(self.k), to_dev(self.v), slot, self.T, kcd, vcd, d))
        out = empty_rows((self.T, self.H, self.D), self.dtype)
        hyb.check(hyb.hyb_paged_attn_prefill_causal(out, to_dev(self.q), kcd, vcd, to_dev(bt), cu_d, ctx_d,
                                                    self.B, self.T, int(self.qlens.max()), d))
        torch.cuda.synchronize()
        return out, to_host(slot), to_host(kcd)


def decode_case(seed, lens, H, D, dtype, block_size=W.BLOCK_SIZE):
    """Decode = one new row per request at position lens[b] - 1."""
    lens = np.asarray(lens, np.int32)
    return PagedCase(seed, np.ones_like(lens), lens - 1, H, D, dtype, block_size)


def decode_gpu(hyb, c, window, bt, max_seq_len=None):
    d = c.dims(hyb, window)
    lens = c.ctx + 1
    msl = int(lens.max()) if max_seq_len is None else max_seq_len
    kcd, vcd = to_dev(c.okc), to_dev(c.ovc)          # this step's rows already appended
    ws_n = hyb.hyb_paged_attn_decode_workspace_size(c.B, msl, d)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device="cuda")
    out = empty_rows((c.B, c.H, c.D), c.dtype)
    hyb.check(hyb.hyb_paged_attn_decode(out, to_dev(c.q), kcd, vcd, to_dev(bt), to_dev(lens), c.B, msl, d,
                                        ws, ws_n))
    torch.cuda.synchronize()
    return out, ws_n
