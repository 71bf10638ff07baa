"""Pins for the CPU oracle: checks against what the pages and the mathematics fix,
never against the oracle's own formula retyped.

Pages: [KV] "推理框架适配Hybrid Model：KV Cache管理与算子调度实战" (icman.com.cn/news/43047).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = int(v)
    return vals


def _f64(a):
    return W.bf16_to_f32(a).astype(np.float64) if a.dtype == np.uint16 else a.astype(np.float64)


def _paged_setup(seed, lens, H, D, dtype, poison=True, slack=1.5, block_size=W.BLOCK_SIZE):
    """Append every row of every request through the oracle's slot mapping into a shuffled
    pool. Returns (pool, kc, vc, k_rows, v_rows, cu)."""
    g = W.rng(seed)
    lens = np.asarray(lens, np.int32)
    pool = W.block_pool(g, lens, slack=slack, block_size=block_size)
    cu = W.cu_from_lens(lens)
    T = int(cu[-1])
    k = W.rows(g, (T, H, D), D, dtype)
    v = W.rows(g, (T, H, D), D, dtype)
    shape = (pool.num_blocks, H, block_size, D)
    if dtype == W.BF16:
        kc = np.full(shape, 0x7FC0 if poison else 0, np.uint16)
    else:
        kc = np.full(shape, np.nan if poison else 0, np.float32)
    vc = kc.copy()
    sm = oracle.slot_mapping(pool.block_tables, cu, block_size=block_size)
    oracle.kv_append(k, v, sm, kc, vc, block_size)
    return pool, kc, vc, k, v, cu, sm


def _sdpa(q, K, V, scale, mask=None):
    """torch's CPU scaled_dot_product_attention in fp64 (library cross-check only)."""
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(K), torch.from_numpy(V),
        attn_mask=None if mask is None else torch.from_numpy(mask), scale=scale).numpy()


# ----------------------------------------------------------------- memory
def test_cache_bytes_worked_example():
    """The page's worked example: 24 Full + 8 Linear layers -> ~103 GB and ~67 MB."""
    g = _read_golden("memory_worked_example.txt")
    tot, full, lin = oracle.cache_bytes(g["L_full"], g["L_linear"], g["H"], g["D"], g["S"],
                                        g["batch"], g["kv_elem_bytes"], g["state_elem_bytes"])
    assert round(full / 1e9) == g["full_printed_GB"]
    assert round(lin / 1e6) == g["linear_printed_MB"]
    assert tot == full + lin


def test_cache_bytes_grow_only_vs_constant():
    """[KV §2.1]: Full KV grows linearly with S; the Linear state does not depend on S."""
    _, f1, l1 = oracle.cache_bytes(3, 1, 4, 16, 1000, 2, 2, 4)
    _, f2, l2 = oracle.cache_bytes(3, 1, 4, 16, 1001, 2, 2, 4)
    _, f3, l3 = oracle.cache_bytes(3, 1, 4, 16, 2000, 2, 2, 4)
    assert l1 == l2 == l3
    assert f3 == 2 * f1 and f2 - f1 == f1 // 1000


# ------------------------------------------------------- append / slots
@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_append_one_slot_per_token_and_bytes_exact(dtype, bs):
    lens = [1, 15, 16, 17, 40, 70]
    H, D = 3, 16
    pool, kc, vc, k, v, cu, sm = _paged_setup(1, lens, H, D, dtype, block_size=bs)
    # exactly one new slot per token, all distinct, all inside the request's own blocks, in
    # position order within each block
    assert len(sm) == sum(lens) and len(set(sm.tolist())) == len(sm)
    for b in range(len(lens)):
        owned = pool.block_tables[b, :pool.blocks_per_req[b]]
        for j, s in enumerate(sm[cu[b]:cu[b + 1]]):
            assert s // bs == owned[j // bs] and s % bs == j % bs
    # the rows appear, byte for byte, at exactly len(sm) slots; every other slot stays poisoned
    written = ~np.isnan(_f64(kc).reshape(pool.num_blocks, H, bs, D)[:, 0, :, 0])
    assert int(written.sum()) == sum(lens)
    for t, s in enumerate(sm):
        assert np.array_equal(kc[s // bs, :, s % bs, :], k[t]) and np.array_equal(vc[s // bs, :, s % bs, :], v[t])


def test_append_skips_minus_one():
    H, D = 2, 16
    k = W.rows(W.rng(2), (3, H, D), D, W.F32)
    kc = np.zeros((4, H, 16, D), np.float32)
    vc = kc.copy()
    oracle.kv_append(k, k, np.array([5, -1, 17], np.int64), kc, vc)
    assert np.array_equal(kc[0, :, 5], k[0]) and np.array_equal(kc[1, :, 1], k[2])
    assert int((kc != 0).any(axis=-1).sum()) == 2 * H


# ------------------------------------------------------------ Full decode
@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_decode_matches_sdpa_on_dense_rows(dtype, bs):
    """Paged decode == dense attention (torch CPU sdpa, fp64) over the rows as generated,
    with 16- and 32-token blocks."""
    lens = [1, 5, 16, 17, 33, 64]
    H, D = 2, 16
    pool, kc, vc, k, v, cu, _ = _paged_setup(3, lens, H, D, dtype, block_size=bs)
    q = W.rows(W.rng(33), (len(lens), H, D), D, dtype)
    scale = 1 / math.sqrt(D)
    out = oracle.full_decode(q, kc, vc, pool.block_tables, lens, scale, block_size=bs)
    for b, n in enumerate(lens):
        K = _f64(k[cu[b]:cu[b + 1]]).transpose(1, 0, 2)      # [H][n][D]
        V = _f64(v[cu[b]:cu[b + 1]]).transpose(1, 0, 2)
        ref = _sdpa(_f64(q[b])[:, None, :], K, V, scale)[:, 0, :]
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-14)


def test_decode_block_permutation_invariance_bit_exact():
    """Paged attention equals contiguous dense attention for ANY block permutation:
    20 seeded pools give bit-identical outputs (same summation order)."""
    lens = [3, 16, 31, 50]
    H, D = 2, 16
    q = W.rows(W.rng(99), (len(lens), H, D), D, W.BF16)
    ref = None
    for seed in range(20):
        g = W.rng(1000)   # identical rows every time ...
        T = sum(lens)
        k = W.rows(g, (T, H, D), D, W.BF16)
        v = W.rows(g, (T, H, D), D, W.BF16)
        pool = W.block_pool(W.rng(seed), lens, slack=2.0)   # ... placed at different blocks
        kc = np.full((pool.num_blocks, H, 16, D), 0x7FC0, np.uint16)
        vc = kc.copy()
        cu = W.cu_from_lens(lens)
        oracle.kv_append(k, v, oracle.slot_mapping(pool.block_tables, cu), kc, vc)
        out = oracle.full_decode(q, kc, vc, pool.block_tables, lens, 0.25)
        if ref is None:
            ref = out
        assert np.array_equal(out, ref)


def test_decode_single_token_returns_v():
    H, D = 2, 16
    pool, kc, vc, k, v, cu, _ = _paged_setup(4, [1, 1], H, D, W.BF16)
    q = W.rows(W.rng(5), (2, H, D), D, W.BF16)
    out = oracle.full_decode(q, kc, vc, pool.block_tables, [1, 1], 0.25)
    assert np.array_equal(out, _f64(v))


def test_decode_equal_keys_gives_mean_of_values():
    H, D, n = 1, 16, 37
    g = W.rng(6)
    k = np.repeat(W.rows(g, (1, H, D), D, W.F32), n, axis=0)
    v = W.rows(g, (n, H, D), D, W.F32)
    pool = W.block_pool(g, [n])
    kc = np.zeros((pool.num_blocks, H, 16, D), np.float32)
    vc = kc.copy()
    oracle.kv_append(k, v, oracle.slot_mapping(pool.block_tables, [0, n]), kc, vc)
    out = oracle.full_decode(W.rows(g, (1, H, D), D, W.F32), kc, vc, pool.block_tables, [n], 0.25)
    np.testing.assert_allclose(out[0, 0], v[:, 0, :].astype(np.float64).mean(0), rtol=1e-12, atol=1e-15)


def test_decode_zero_length_gives_zero():
    H, D = 2, 16
    pool, kc, vc, *_ = _paged_setup(7, [4, 1], H, D, W.F32)
    q = W.rows(W.rng(8), (2, H, D), D, W.F32)
    out = oracle.full_decode(q, kc, vc, pool.block_tables, [0, 1], 0.25)
    assert not out[0].any()


# ---------------------------------------------------------- Full prefill
@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("ctx", [[0, 0], [16, 5]])
def test_prefill_matches_causal_sdpa(ctx, bs):
    """Causal prefill (queries at absolute positions ctx + j see keys p <= position)
    == torch CPU sdpa with an explicit inclusive causal mask, fp64; 16- and 32-token blocks."""
    H, D = 2, 16
    qlens = [5, 37]
    tot = [c + n for c, n in zip(ctx, qlens)]
    pool, kc, vc, k, v, cu_all, _ = _paged_setup(9, tot, H, D, W.BF16, block_size=bs)
    g = W.rng(10)
    cuq = W.cu_from_lens(qlens)
    q = W.rows(g, (int(cuq[-1]), H, D), D, W.BF16)
    scale = 1 / math.sqrt(D)
    out = oracle.full_prefill(q, kc, vc, pool.block_tables, cuq, ctx, scale, block_size=bs)
    for b in range(2):
        K = _f64(k[cu_all[b]:cu_all[b + 1]]).transpose(1, 0, 2)
        V = _f64(v[cu_all[b]:cu_all[b + 1]]).transpose(1, 0, 2)
        Q = _f64(q[cuq[b]:cuq[b + 1]]).transpose(1, 0, 2)
        pos = ctx[b] + np.arange(qlens[b])
        mask = np.where(np.arange(tot[b])[None, :] <= pos[:, None], 0.0, -np.inf)
        ref = _sdpa(Q, K, V, scale, mask).transpose(1, 0, 2)
        np.testing.assert_allclose(out[cuq[b]:cuq[b + 1]], ref, rtol=1e-12, atol=1e-14)
    # row subset gives the same rows
    rows = np.array([0, 4, 5, 41], np.int32)
    np.testing.assert_array_equal(oracle.full_prefill(q, kc, vc, pool.block_tables, cuq, ctx, scale, rows,
                                                      block_size=bs), out[rows])


# ------------------------------------------------- sliding-window Full attention
# [KV §1.3] names sliding-window attention as the model-side alternative to paged KV:
# a query at absolute position i sees only the keys at positions i - W < p <= i.
@pytest.mark.parametrize("window", [1, 5, 16, 17, 40])
def test_window_decode_matches_banded_sdpa(window):
    lens = [1, 5, 16, 17, 33, 64]
    H, D = 2, 16
    pool, kc, vc, k, v, cu, _ = _paged_setup(21, lens, H, D, W.BF16)
    q = W.rows(W.rng(22), (len(lens), H, D), D, W.BF16)
    scale = 1 / math.sqrt(D)
    out = oracle.full_decode(q, kc, vc, pool.block_tables, lens, scale, window=window)
    for b, n in enumerate(lens):
        K = _f64(k[cu[b]:cu[b + 1]]).transpose(1, 0, 2)
        V = _f64(v[cu[b]:cu[b + 1]]).transpose(1, 0, 2)
        mask = np.where(np.arange(n)[None, :] > n - 1 - window, 0.0, -np.inf)
        ref = _sdpa(_f64(q[b])[:, None, :], K, V, scale, mask)[:, 0, :]
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("window,ctx", [(1, [0, 0]), (7, [16, 5]), (16, [0, 40]), (33, [16, 5])])
def test_window_prefill_matches_banded_causal_sdpa(window, ctx):
    H, D = 2, 16
    qlens = [5, 37]
    tot = [c + n for c, n in zip(ctx, qlens)]
    pool, kc, vc, k, v, cu_all, _ = _paged_setup(23, tot, H, D, W.BF16)
    cuq = W.cu_from_lens(qlens)
    q = W.rows(W.rng(24), (int(cuq[-1]), H, D), D, W.BF16)
    scale = 1 / math.sqrt(D)
    out = oracle.full_prefill(q, kc, vc, pool.block_tables, cuq, ctx, scale, window=window)
    for b in range(2):
        K = _f64(k[cu_all[b]:cu_all[b + 1]]).transpose(1, 0, 2)
        V = _f64(v[cu_all[b]:cu_all[b + 1]]).transpose(1, 0, 2)
        Q = _f64(q[cuq[b]:cuq[b + 1]]).transpose(1, 0, 2)
        pos = ctx[b] + np.arange(qlens[b])
        p = np.arange(tot[b])[None, :]
        mask = np.where((p <= pos[:, None]) & (p > pos[:, None] - window), 0.0, -np.inf)
        ref = _sdpa(Q, K, V, scale, mask).transpose(1, 0, 2)
        np.testing.assert_allclose(out[cuq[b]:cuq[b + 1]], ref, rtol=1e-12, atol=1e-14)


def test_window_covering_every_key_is_full_attention_bit_exact():
    H, D = 2, 16
    lens = [3, 16, 31]
    pool, kc, vc, k, v, cu, _ = _paged_setup(25, lens, H, D, W.F32)
    q = W.rows(W.rng(26), (len(lens), H, D), D, W.F32)
    full = oracle.full_decode(q, kc, vc, pool.block_tables, lens, 0.25)
    for window in (31, 32, 1000):
        assert np.array_equal(oracle.full_decode(q, kc, vc, pool.block_tables, lens, 0.25,
                                                 window=window), full)
    qp = W.rows(W.rng(27), (int(cu[-1]), H, D), D, W.F32)
    fullp = oracle.full_prefill(qp, kc, vc, pool.block_tables, cu, [0, 0, 0], 0.25)
    assert np.array_equal(oracle.full_prefill(qp, kc, vc, pool.block_tables, cu, [0, 0, 0], 0.25,
                                              window=31), fullp)


def test_window_one_returns_own_value():
    """W = 1: each query sees only its own position, so the output is that value row."""
    H, D = 2, 16
    lens = [4, 20]
    pool, kc, vc, k, v, cu, _ = _paged_setup(28, lens, H, D, W.BF16)
    q = W.rows(W.rng(29), (int(cu[-1]), H, D), D, W.BF16)
    out = oracle.full_prefill(q, kc, vc, pool.block_tables, cu, [0, 0], 0.25, window=1)
    assert np.array_equal(out, _f64(v))
    qd = W.rows(W.rng(30), (2, H, D), D, W.BF16)
    outd = oracle.full_decode(qd, kc, vc, pool.block_tables, lens, 0.25, window=1)
    assert np.array_equal(outd, _f64(v[cu[1:] - 1]))


def test_prefill_last_row_equals_decode_on_same_prefix():
    H, D = 2, 16
    pool, kc, vc, k, v, cu, _ = _paged_setup(11, [20, 7], H, D, W.BF16)
    q = W.rows(W.rng(12), (27, H, D), D, W.BF16)
    pre = oracle.full_prefill(q, kc, vc, pool.block_tables, cu, [0, 0], 0.25)
    dec = oracle.full_decode(q[[19, 26]], kc, vc, pool.block_tables, [20, 7], 0.25)
    assert np.array_equal(pre[[19, 26]], dec)


# ------------------------------------------------------------ Linear
def test_linear_zero_state_one_token_is_outer_product():
    """[KV §2.1]: a zeroed state plus one token holds exactly k (outer) v; the output is
    q.S = (q.k) v (state updated before the output is read)."""
    H, D = 3, 16
    g = W.rng(13)
    q, k, v = (W.rows(g, (1, H, D), D, W.BF16) for _ in range(3))
    out, st = oracle.linear_recurrence(q, k, v, [0, 1])
    K, V, Q = _f64(k[0]), _f64(v[0]), _f64(q[0])
    for h in range(H):
        assert np.array_equal(st[0, h], np.outer(K[h], V[h]))      # exact: bf16 x bf16 fits fp64
        np.testing.assert_allclose(out[0, h], (Q[h] @ K[h]) * V[h], rtol=1e-13, atol=1e-16)
        # not the transposed orientation v k^T and not the pre-update (zero) output
        assert not np.allclose(out[0, h], (Q[h] @ V[h]) * K[h])


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_linear_matches_textbook_matrix_form(dtype):
    """O = Q S0 + tril(Q K^T) V and S_T = S0 + K^T V (numpy matmul, fp64)."""
    H, D = 2, 16
    lens = [1, 9, 40]
    g = W.rng(14)
    cu = W.cu_from_lens(lens)
    T = int(cu[-1])
    q, k, v = (W.rows(g, (T, H, D), D, dtype) for _ in range(3))
    pool = W.synthetic_state(g, 4, H, D, np.array([10, 20, 30, 40]))
    slots = np.array([2, 0, 3], np.int32)
    reset = np.array([0, 1, 0], np.uint8)
    out, st = oracle.linear_recurrence(q, k, v, cu, pool, slots, reset)
    for b in range(3):
        for h in range(H):
            Q, K, V = (_f64(a[cu[b]:cu[b + 1], h]) for a in (q, k, v))
            S0 = np.zeros((D, D)) if reset[b] else pool[slots[b], h].astype(np.float64)
            ref_o = Q @ S0 + np.tril(Q @ K.T) @ V
            ref_s = S0 + K.T @ V
            np.testing.assert_allclose(out[cu[b]:cu[b + 1], h], ref_o, rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(st[b, h], ref_s, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("C", [1, 2, 3, 5, 7, 16, 64, 128, 300])
def test_linear_chunked_equals_recurrence(C):
    """Token-by-token recurrence == chunk form for every chunk size."""
    H, D = 2, 16
    lens = [1, 63, 64, 65, 130, 300]
    g = W.rng(15)
    cu = W.cu_from_lens(lens)
    T = int(cu[-1])
    q, k, v = (W.rows(g, (T, H, D), D, W.BF16) for _ in range(3))
    pool = W.synthetic_state(g, len(lens), H, D, np.full(len(lens), 50))
    slots = np.arange(len(lens), dtype=np.int32)[::-1].copy()
    reset = np.array([1, 0, 1, 0, 1, 0], np.uint8)
    o1, s1 = oracle.linear_recurrence(q, k, v, cu, pool, slots, reset)
    o2, s2 = oracle.linear_chunked(q, k, v, cu, C, None, pool, slots, reset)
    scale_o = np.abs(o1).max()
    assert np.abs(o1 - o2).max() <= 1e-12 * scale_o
    assert np.abs(s1 - s2).max() <= 1e-12 * np.abs(s1).max()


def test_linear_chunked_unaligned_start_and_split_calls():
    """Prefill(n) carried into prefill(m) == prefill(n+m), chunk boundaries at absolute
    positions; also holds when the split point is not chunk-aligned."""
    H, D, C = 2, 16, 8
    n_tot = 45
    g = W.rng(16)
    q, k, v = (W.rows(g, (n_tot, H, D), D, W.BF16) for _ in range(3))
    o_all, s_all = oracle.linear_chunked(q, k, v, [0, n_tot], C)
    for split in (8, 13, 40):
        o1, s1 = oracle.linear_chunked(q[:split], k[:split], v[:split], [0, split], C)
        pool = s1.astype(np.float32)            # carried state (fp32 storage)
        o2, s2 = oracle.linear_chunked(q[split:], k[split:], v[split:], [0, n_tot - split], C,
                                       ctx_lens=[split], state_pool=pool, state_slots=[0])
        np.testing.assert_allclose(np.concatenate([o1, o2]), o_all, rtol=1e-6, atol=1e-7)
        np.testing.assert_allclose(s2, s_all, rtol=1e-6, atol=1e-7)


def test_linear_prefill_then_decode_equals_longer_prefill():
    H, D = 2, 16
    n, m = 20, 4
    g = W.rng(17)
    q, k, v = (W.rows(g, (n + m, H, D), D, W.F32) for _ in range(3))
    o_all, s_all = oracle.linear_recurrence(q, k, v, [0, n + m])
    _, s = oracle.linear_recurrence(q[:n], k[:n], v[:n], [0, n])
    outs = []
    state = s.astype(np.float64)
    for t in range(n, n + m):
        o, state = oracle.linear_recurrence(q[t:t + 1], k[t:t + 1], v[t:t + 1], [0, 1],
                                            state_pool=state.astype(np.float32), state_slots=[0])
        outs.append(o[0])
    np.testing.assert_allclose(np.stack(outs), o_all[n:], rtol=1e-5, atol=1e-6)


def test_linear_state_size_constant_and_reset_forgets():
    """State bytes do not depend on sequence length [KV §2.1]; a reset slot ignores whatever
    the previous request left there [KV §2.3]."""
    H, D = 2, 16
    g = W.rng(18)
    q, k, v = (W.rows(g, (50, H, D), D, W.F32) for _ in range(3))
    _, s_short = oracle.linear_recurrence(q[:3], k[:3], v[:3], [0, 3])
    _, s_long = oracle.linear_recurrence(q, k, v, [0, 50])
    assert s_short.nbytes == s_long.nbytes
    junk = W.synthetic_state(g, 1, H, D, np.array([99]))
    o_a, s_a = oracle.linear_recurrence(q, k, v, [0, 50], junk, [0], np.array([1], np.uint8))
    assert np.array_equal(o_a, oracle.linear_recurrence(q, k, v, [0, 50])[0])


# ------------------------------------------- 16-bit linear state (state-precision study)
def _round16(x32, state_dtype):
    """Library rounding of fp32 values to bf16 (torch) or fp16 (numpy), as uint16 bits."""
    if state_dtype == 1:
        return torch.from_numpy(np.ascontiguousarray(x32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return np.ascontiguousarray(x32).astype(np.float16).view(np.uint16)


def _widen16(u, state_dtype):
    u = np.ascontiguousarray(u)
    return W.bf16_to_f32(u).astype(np.float64) if state_dtype == 1 else u.view(np.float16).astype(np.float64)


@pytest.mark.parametrize("state_dtype", [1, 2])
def test_lowp_state_one_token_is_rounded_product(state_dtype):
    """Zero state + one token: S_ij = round16(k_i v_j), the fp32 product (exact for bf16
    inputs) rounded by torch (bf16) or numpy (fp16); the output is q . S on that rounded
    state (numpy, fp64)."""
    H, D = 2, 16
    g = W.rng(40)
    q, k, v = (W.rows(g, (1, H, D), D, W.BF16) for _ in range(3))
    out, st = oracle.linear_recurrence_lowp(q, k, v, [0, 1], state_dtype)
    kf, vf = W.bf16_to_f32(k[0]), W.bf16_to_f32(v[0])
    prod = (kf[:, :, None] * vf[:, None, :]).astype(np.float32)
    ref_st = _round16(prod, state_dtype)
    assert np.array_equal(st[0], ref_st)
    ref_out = np.einsum("hi,hij->hj", W.bf16_to_f32(q[0]).astype(np.float64), _widen16(ref_st, state_dtype))
    np.testing.assert_allclose(out[0], ref_out, rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("state_dtype", [1, 2])
def test_lowp_state_exact_when_representable(state_dtype):
    """Inputs in {0, +-1/4, +-1/2} keep every product and partial state a multiple of 1/16
    below 1 in magnitude, exact in bf16 and fp16: the 16-bit recurrence then equals the
    fp64 recurrence exactly (states and outputs), over two requests of three tokens."""
    H, D, T = 2, 8, 6
    g = np.random.default_rng(41)
    mk = lambda: (g.integers(-2, 3, (T, H, D)) / 4.0).astype(np.float32)
    q, k, v = mk(), mk(), mk()
    cu = [0, 3, 6]
    out, st = oracle.linear_recurrence_lowp(q, k, v, cu, state_dtype)
    ref_out, ref_st = oracle.linear_recurrence(q, k, v, cu)
    assert np.array_equal(_widen16(st, state_dtype), ref_st)
    assert np.array_equal(out, ref_out)


def test_lowp_bf16_state_drops_updates_below_half_an_ulp():
    """bf16 keeps 8 significant bits: at S = 256 an update k v = 0.5 is below half the
    spacing (2) and the state stays 256; fp16 (spacing 0.25 at 256) keeps 256.5."""
    one = lambda x: np.full((1, 1, 1), x, np.float32)
    for sd, start, expect in ((1, 0x4380, 256.0), (2, 0x5C00, 256.5)):
        pool = np.full((1, 1, 1, 1), start, np.uint16)
        out, st = oracle.linear_recurrence_lowp(one(1.0), one(1.0), one(0.5), [0, 1], sd,
                                                state_pool=pool, state_slots=[0])
        assert _widen16(st, sd)[0, 0, 0, 0] == expect and out[0, 0, 0] == expect
