"""Shared helpers of the GPU parity tests: host <-> device copies of the seeded inputs,
the tolerance rules the tests apply, and paged cases with peaked attention scores.

Tolerances (floating point). A bf16/fp32 attention output passes when both hold:
  * every element: |gpu - ref| <= 2e-2 + 1e-2 * |ref| (the allclose reading of
    "2e-2 max-abs / 1e-2 relative");
  * every output row (the D values of one (token, head)): max|gpu - ref| <=
    1e-2 * max|ref| over that row. This is the scale-relative half of the same rule; it
    is what holds a decode output of size 1e-3 (long rows average many value rows) to
    the bound, where the absolute 2e-2 alone would accept anything.
fp32 linear states pass when, for every (request, head) matrix, max|gpu - ref| <=
1e-3 * max|ref|. Integer and byte results (slots, cache images) must be identical.
Every check records the achieved row-relative error; the session prints the worst per test.
"""
import math
import os

import numpy as np
import torch

import oracle
import workloads as W

OUT_ATOL = 2e-2
OUT_REL = 1e-2
ROW_REL = 1e-2
STATE_REL = 1e-3

# (test id, what, worst row-relative error, max abs error) of every output check
RECORDS = []


def to_dev(a: np.ndarray, dtype_code: int | None = None, device="cuda"):
    """numpy -> CUDA tensor. uint16 arrays are bf16 bit patterns."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def lin_ws(device="cuda"):
    """(workspace, bytes) for one hyb_linear_attn_chunked_prefill call: a fresh device
    buffer of the size the library asks for (its contents need no initialisation)."""
    import paged_kv_linear_gb300 as hyb
    n = hyb.hyb_linear_attn_chunked_prefill_workspace_size()
    return torch.empty(n, dtype=torch.uint8, device=device), n


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


def out_close_report(gpu, ref):
    """(elementwise ok, rows ok, worst row-relative error, max abs error) of the output rule.
    A row whose reference is all zero must be exactly zero."""
    g = as_f64(gpu)
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    if not g.size:
        return True, True, 0.0, 0.0
    if not np.isfinite(g).all():
        return False, False, math.inf, math.inf
    err = np.abs(g - ref)
    elem_ok = bool((err <= OUT_ATOL + OUT_REL * np.abs(ref)).all())
    e2 = err.reshape(-1, err.shape[-1]).max(axis=1)
    m2 = np.abs(ref).reshape(-1, ref.shape[-1]).max(axis=1)
    rows_ok = bool((e2 <= ROW_REL * m2).all())
    rel = np.where(m2 > 0, e2 / np.where(m2 > 0, m2, 1.0), np.where(e2 > 0, math.inf, 0.0))
    return elem_ok, rows_ok, float(rel.max()), float(err.max())


def assert_out_close(gpu, ref, what="output"):
    """The output rule (module docstring): elementwise |g - r| <= 2e-2 + 1e-2 |r| and, per
    output row, max|g - r| <= 1e-2 max|r|; every value finite. Records and returns the worst
    row-relative error."""
    g = as_f64(gpu)
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    if not g.size:
        return 0.0
    elem_ok, rows_ok, rel, abs_err = out_close_report(g, ref)
    RECORDS.append((os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0], what, rel, abs_err))
    print(f"{what}: worst row-relative error {rel:.3e} (bound {ROW_REL:g}), max abs error {abs_err:.3e}")
    if not elem_ok:
        err = np.abs(g - ref)
        lim = OUT_ATOL + OUT_REL * np.abs(ref)
        worst = int(np.argmax(err - lim))
        raise AssertionError(f"{what}: |err| {err.flat[worst]:.3e} > {lim.flat[worst]:.3e} "
                             f"at ref {ref.flat[worst]:.3e}; max abs err {abs_err:.3e}")
    assert rows_ok, f"{what}: a row's max|err| exceeds {ROW_REL:g} x its max|ref| (worst ratio {rel:.3e})"
    return rel


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


class Peaked:
    """Rows of a paged case whose attention scores follow a chosen profile along the key
    position. Queries are alpha * u[h] plus N(0,1)/sqrt(D) noise; the key at absolute
    position p of request b carries f(p) / (scale * alpha) along u[h], so every query's
    score against it is f(p) (natural-log units) plus noise of about 0.06 at D = 128.
    Values are N(0,1)/sqrt(D). Profiles over a request of n keys, amplitude A:
      rise    A p / (n - 1): the running max grows through every key tile and split
      fall    A (1 - p / (n - 1)): the first tile holds the max; later splits weigh e^-A
      waves   A/2 (1 + sin(2 pi p / 1536)): equal maxima in many splits
      spikes  A on 8 random keys of the request, 0 elsewhere: the output is their values' mean
      hot     no direction: q x 24, k x 16 (score std about 3 at D = 128)
    """

    PROFILES = ("rise", "fall", "waves", "spikes", "hot")

    def __init__(self, profile, g, H, D, dtype, total_lens, A=40.0, alpha=8.0):
        assert profile in self.PROFILES, profile
        self.profile, self.g, self.H, self.D, self.dtype = profile, g, H, D, dtype
        self.A, self.alpha, self.scale = float(A), float(alpha), 1 / math.sqrt(D)
        self.n = np.asarray(total_lens, np.int64)
        self.u = W.unit_dirs(g, H, D)
        self.spike = [np.zeros(int(n), bool) for n in self.n]
        for b, n in enumerate(self.n):
            if n:
                self.spike[b][g.choice(int(n), min(8, int(n)), replace=False)] = True

    def f(self, pos, req):
        """Score offset of the keys at absolute positions pos of requests req."""
        pos = np.asarray(pos, np.float64)
        span = np.maximum(self.n[req] - 1, 1).astype(np.float64)
        if self.profile == "rise":
            return self.A * pos / span
        if self.profile == "fall":
            return self.A * (1 - pos / span)
        if self.profile == "waves":
            return self.A * 0.5 * (1 + np.sin(2 * np.pi * pos / 1536.0))
        if self.profile == "spikes":
            return np.array([self.A if self.spike[b][int(p)] else 0.0 for p, b in zip(pos, req)])
        return np.zeros(len(pos))

    def queries(self, T):
        if self.profile == "hot":
            return W.directed_rows(self.g, np.zeros(T), self.u, self.D, self.dtype, noise=24.0)
        return W.directed_rows(self.g, np.full(T, self.alpha), self.u, self.D, self.dtype)

    def keys(self, pos, req):
        if self.profile == "hot":
            return W.directed_rows(self.g, np.zeros(len(pos)), self.u, self.D, self.dtype, noise=16.0)
        coef = self.f(pos, req) / (self.scale * self.alpha)
        return W.directed_rows(self.g, coef, self.u, self.D, self.dtype)

    def values(self, T):
        return W.rows(self.g, (T, self.H, self.D), self.D, self.dtype)


def _positions(lens, start=None):
    """(absolute positions, request index) of rows packed request after request."""
    lens = np.asarray(lens, np.int64)
    start = np.zeros_like(lens) if start is None else np.asarray(start, np.int64)
    pos = np.concatenate([np.arange(s, s + n) for s, n in zip(start, lens)] + [np.zeros(0, np.int64)])
    req = np.repeat(np.arange(len(lens)), lens)
    return pos, req


class PagedCase:
    """Requests with a cached prefix (ctx rows, written by the oracle into a poisoned pool)
    and this call's q/k/v rows (qlens per request). peaked = a Peaked profile name draws
    structured scores instead of N(0,1)/sqrt(D) rows."""

    def __init__(self, seed, qlens, ctx, H, D, dtype, block_size=W.BLOCK_SIZE, peaked=None):
        g = W.rng(seed)
        self.qlens = np.asarray(qlens, np.int32)
        self.ctx = np.asarray(ctx, np.int32)
        self.B, self.H, self.D, self.dtype = len(self.qlens), H, D, dtype
        self.bs = block_size
        self.pool = W.block_pool(g, self.qlens + self.ctx, block_size=block_size)
        cu_ctx = W.cu_from_lens(self.ctx)
        self.gen = Peaked(peaked, g, H, D, dtype, self.qlens + self.ctx) if peaked else None
        if self.gen:
            kp = self.gen.keys(*_positions(self.ctx))
            vp = self.gen.values(int(cu_ctx[-1]))
        else:
            kp, vp = (W.rows(g, (int(cu_ctx[-1]), H, D), D, dtype) for _ in range(2))
        self.kc = poisoned_pool(self.pool.num_blocks, H, D, dtype, block_size)
        self.vc = self.kc.copy()
        oracle.kv_append(kp, vp, oracle.slot_mapping(self.pool.block_tables, cu_ctx, block_size=block_size),
                         self.kc, self.vc, block_size)
        self.cu = W.cu_from_lens(self.qlens)
        self.T = int(self.cu[-1])
        if self.gen:
            self.q = self.gen.queries(self.T)
            self.k = self.gen.keys(*_positions(self.qlens, self.ctx))
            self.v = self.gen.values(self.T)
        else:
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


def decode_case(seed, lens, H, D, dtype, block_size=W.BLOCK_SIZE, peaked=None):
    """Decode = one new row per request at position lens[b] - 1."""
    lens = np.asarray(lens, np.int32)
    return PagedCase(seed, np.ones_like(lens), lens - 1, H, D, dtype, block_size, peaked)


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
