"""The output parity rule can fail: on CPU, with the oracle as the reference.

A decode output over n keys averages many value rows, so its size falls like 1/sqrt(n)
(about 6e-3 at n = 4096 with N(0,1)/sqrt(D) inputs) and the absolute 2e-2 half of the
rule alone accepts anything there. The row-relative half (max|g - r| <= 1e-2 max|r| per
output row) must reject a wrong result at any size. Here it rejects, on n = 4096 rows with
peaked scores ("推理框架适配Hybrid Model：KV Cache管理与算子调度实战", §3.5 validates
against a reference as the length grows):
  * the output scaled by 0.98, an all-zero output, the uniform-softmax mean of V;
  * a tiled online softmax that skips the rescale of the running sum when the max grows
    (the lazy-rescale branch of the tensor-core prefill), and a split-K combine that
    ignores the splits' maxima (the decode's log-sum-exp merge).
The same tiled softmax done right passes. With N(0,1)/sqrt(D) inputs the scores' spread
is about 1/D, the softmax is uniform to about 1 %, and the uniform mean lands at the bound
itself: that blind spot is why the GPU parity tests also run the peaked profiles.
"""
import math

import numpy as np
import pytest

import workloads as W
from gpu_helpers import ROW_REL, as_f64, decode_case, out_close_report

LOG2E = 1.4426950408889634


def _passes(gpu, ref):
    elem_ok, rows_ok, _, _ = out_close_report(gpu, ref)
    return elem_ok and rows_ok


def _dense(c, b, h, which):
    """Rows 0..n-1 of request b, head h, gathered from the oracle's cache image."""
    n = int(c.ctx[b]) + 1
    pool = c.okc if which == "k" else c.ovc
    blocks = c.pool.block_tables[b, :(n + c.bs - 1) // c.bs]
    return as_f64(pool[blocks, h].reshape(-1, c.D)[:n])


def _tiled(c, rescale=True, combine_max=True, tile=128, split=512):
    """Decode by splits of `split` keys, each an online softmax over `tile`-key tiles that
    rescales only when the running max grows by more than 2^8 (log2 units)."""
    out = np.zeros((c.B, c.H, c.D))
    q = as_f64(c.q)
    for b in range(c.B):
        for h in range(c.H):
            K, V = _dense(c, b, h, "k"), _dense(c, b, h, "v")
            s = K @ q[b, h] * c.scale * LOG2E
            parts = []
            for s0 in range(0, len(s), split):
                m, l, acc = -math.inf, 0.0, np.zeros(c.D)
                for t0 in range(s0, min(len(s), s0 + split), tile):
                    x = s[t0:min(len(s), s0 + split, t0 + tile)]
                    mn = max(m, x.max())
                    if m == -math.inf or mn > m + 8:
                        if m != -math.inf and rescale:
                            alpha = 2.0 ** (m - mn)
                            acc, l = acc * alpha, l * alpha
                        m = mn
                    p = 2.0 ** (x - m)
                    l += p.sum()
                    acc += p @ V[t0:t0 + len(x)]
                parts.append((m, l, acc))
            M = max(pm for pm, _, _ in parts)
            w = [2.0 ** (pm - M) if combine_max else 1.0 for pm, _, _ in parts]
            out[b, h] = sum(wi * a for wi, (_, _, a) in zip(w, parts)) / sum(wi * pl for wi, (_, pl, _) in zip(w, parts))
    return out


def _uniform_mean(c):
    return np.stack([np.stack([_dense(c, b, h, "v").mean(axis=0) for h in range(c.H)]) for b in range(c.B)])


@pytest.fixture(scope="module", params=["rise", "waves", "spikes", "hot"])
def peaked(request):
    c = decode_case(90, [4096, 4096, 2500], 4, 128, W.BF16, peaked=request.param)
    return c, c.decode_ref()


@pytest.fixture(scope="module")
def plain():
    c = decode_case(91, [4096, 4096], 4, 128, W.BF16)
    return c, c.decode_ref()


def test_rule_accepts_the_reference_rounded_to_bf16(peaked, plain):
    for c, ref in (peaked, plain):
        assert _passes(W.bf16_round(ref.astype(np.float32)), ref)


def test_rule_rejects_scaled_and_zero_outputs(peaked, plain):
    for c, ref in (peaked, plain):
        assert not _passes(W.bf16_round((0.98 * ref).astype(np.float32)), ref)
        assert not _passes(np.zeros_like(ref), ref)
        # the absolute half alone would have accepted the zeros: outputs are that small
        assert np.abs(ref).max() < 2e-2 or c.gen is not None


def test_rule_rejects_uniform_softmax_mean_on_peaked_scores(peaked):
    c, ref = peaked
    assert not _passes(_uniform_mean(c), ref)


def test_plain_inputs_barely_separate_softmax_from_uniform_mean(plain):
    """The blind spot the peaked profiles close: with N(0,1)/sqrt(D) inputs the softmax
    weights differ from uniform by about 1/D, so the uniform mean lands within about 1 %
    of the reference, at the bound itself: such inputs cannot tell a softmax bug apart."""
    c, ref = plain
    _, _, rel, _ = out_close_report(_uniform_mean(c), ref)
    assert rel < 2 * ROW_REL


def test_tiled_online_softmax_passes_and_its_mutants_fail(peaked):
    c, ref = peaked
    assert _passes(_tiled(c), ref)
    if c.gen.profile in ("rise", "spikes", "waves"):     # maxima that move between tiles
        assert not _passes(_tiled(c, rescale=False), ref)
    assert not _passes(_tiled(c, combine_max=False), ref)
