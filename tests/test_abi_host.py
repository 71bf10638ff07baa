"""Host-only checks of the C-ABI library: it loads, exports every entry point that
include/hyb.h declares, and rejects bad arguments before touching the GPU."""
import ctypes as C
import os
import re

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def hyb():
    from paged_kv_linear_gb300 import _build
    _build.build()
    import paged_kv_linear_gb300 as hyb
    return hyb


def declared_entry_points():
    src = open(os.path.join(ROOT, "include", "hyb.h"), encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(hyb_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol(hyb):
    names = declared_entry_points()
    assert len(names) >= 12
    L = C.CDLL(hyb.LIB)
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/hyb.h but not exported"


def test_cache_bytes_matches_oracle_and_worked_example(hyb):
    args = (24, 8, 32, 128, 32768, 8, 2, 2)
    assert hyb.hyb_cache_bytes(*args) == oracle.cache_bytes(*args)
    tot, full, lin = hyb.hyb_cache_bytes(*args)
    assert round(full / 1e9) == 103 and round(lin / 1e6) == 67


def test_status_strings(hyb):
    for s in range(5):
        assert hyb.status_string(s)
    assert "unknown" in hyb.status_string(99)


def test_bad_arguments_rejected_before_launch(hyb):
    d = hyb.dims(32, 128, 100, 8)
    fake = 1 << 20      # aligned, never dereferenced: validation fails first
    # null pointers
    assert hyb.hyb_paged_kv_append(None, fake, fake, 4, fake, fake + 256, d, 0) == hyb.HYB_ERR_INVALID_ARG
    # misaligned data pointer
    assert hyb.hyb_paged_kv_append(fake + 2, fake, fake, 4, fake, fake + 256, d, 0) == hyb.HYB_ERR_INVALID_ARG
    # the same pool passed as K and V
    assert hyb.hyb_paged_kv_append(fake, fake, fake, 4, fake, fake, d, 0) == hyb.HYB_ERR_INVALID_ARG
    # block sizes other than a power of two from 16 to 256
    for bs in (8, 24, 48, 512):
        dbs = hyb.dims(32, 128, 100, 8, block_size=bs)
        assert hyb.hyb_paged_kv_append(fake, fake, fake, 4, fake, fake + 256, dbs, 0) == hyb.HYB_ERR_UNSUPPORTED
    # max_seq_len is bounded by max_blocks_per_seq x block_size
    d32 = hyb.dims(32, 128, 100, 8, block_size=32)
    assert hyb.hyb_paged_attn_decode(fake, fake, fake, fake, fake, fake, 2, 257, d32, fake, 1 << 20, 0) == hyb.HYB_ERR_INVALID_ARG
    # pools whose rows (blocks x heads x block size) overflow int32
    dbig = hyb.dims(32, 128, 1 << 20, 8, block_size=128)
    assert hyb.hyb_paged_kv_append(fake, fake, fake, 4, fake, fake + 256, dbig, 0) == hyb.HYB_ERR_UNSUPPORTED
    # head_dim without a kernel
    d7 = hyb.dims(4, 24, 100, 8)
    assert hyb.hyb_paged_attn_decode(fake, fake, fake, fake, fake, fake, 2, 32, d7, None, 0, 0) == hyb.HYB_ERR_UNSUPPORTED
    # more rows than the decode grid takes (grid.y = rows <= 65535)
    assert hyb.hyb_paged_attn_decode(fake, fake, fake, fake, fake, fake, 65536, 32, d, fake, 1 << 20, 0) == hyb.HYB_ERR_UNSUPPORTED
    # max_seq_len beyond the block table's capacity (8 blocks x 16)
    assert hyb.hyb_paged_attn_decode(fake, fake, fake, fake, fake, fake, 2, 129, d, fake, 1 << 20, 0) == hyb.HYB_ERR_INVALID_ARG
    # workspace too small for a split sequence
    need = hyb.hyb_paged_attn_decode_workspace_size(2, 128, hyb.dims(32, 128, 100, 64))
    d64 = hyb.dims(32, 128, 100, 64)
    need = hyb.hyb_paged_attn_decode_workspace_size(2, 1024, d64)
    assert need > 0
    assert hyb.hyb_paged_attn_decode(fake, fake, fake, fake, fake, fake, 2, 1024, d64, fake, need - 16, 0) == hyb.HYB_ERR_INVALID_ARG
    # fused append + decode: no k / misaligned k / misaligned slot mapping / K and V the same
    # pool / small workspace (a null slot mapping is valid: positions from the block table)
    da = lambda k, slot, kc, vc, ws_b: hyb.hyb_paged_attn_decode_append(
        fake, fake, k, fake, slot, kc, vc, fake, fake, 2, 1024, d64, fake, ws_b, 0)
    assert da(None, fake, fake, fake + 256, need) == hyb.HYB_ERR_INVALID_ARG
    assert da(None, None, fake, fake + 256, need) == hyb.HYB_ERR_INVALID_ARG
    assert da(fake + 2, fake, fake, fake + 256, need) == hyb.HYB_ERR_INVALID_ARG
    assert da(fake, fake + 4, fake, fake + 256, need) == hyb.HYB_ERR_INVALID_ARG
    assert da(fake, fake, fake, fake, need) == hyb.HYB_ERR_INVALID_ARG
    assert da(fake, fake, fake, fake + 256, need - 16) == hyb.HYB_ERR_INVALID_ARG
    assert hyb.hyb_paged_attn_decode_append(fake, fake, fake, fake, fake, fake, fake + 256, fake, fake, 0, 1,
                                            d64, None, 0, 0) == hyb.HYB_OK   # empty batch: nothing to do
    # linear step: no slots / bad dtype / unsupported D
    assert hyb.hyb_linear_attn_step(fake, fake, fake, fake, fake, 0, fake, 2, 4, 128, 1, 0) == hyb.HYB_ERR_INVALID_ARG
    assert hyb.hyb_linear_attn_step(fake, fake, fake, fake, fake, 4, fake, 2, 4, 128, 7, 0) == hyb.HYB_ERR_INVALID_ARG
    assert hyb.hyb_linear_attn_step(fake, fake, fake, fake, fake, 4, fake, 2, 4, 48, 1, 0) == hyb.HYB_ERR_UNSUPPORTED
    # chunked linear prefill: chunk size 0; the handoff workspace missing, short or misaligned
    n_lw = hyb.hyb_linear_attn_chunked_prefill_workspace_size()
    assert n_lw == 8 * (1 + 256)                 # one epoch word and one flag per CTA (<= 256 CTAs)
    lp = lambda C, ws, n, B=2: hyb.hyb_linear_attn_chunked_prefill(fake, fake, fake, fake, fake, None, fake, 4, fake,
                                                                   None, B, 128, 64, 4, 128, C, 1, ws, n, 0)
    assert lp(0, fake, n_lw) == hyb.HYB_ERR_INVALID_ARG
    assert lp(64, None, 0) == hyb.HYB_ERR_INVALID_ARG
    assert lp(64, fake, n_lw - 8) == hyb.HYB_ERR_INVALID_ARG
    assert lp(64, fake + 4, n_lw) == hyb.HYB_ERR_INVALID_ARG
    assert lp(64, None, 0, B=0) == hyb.HYB_OK    # empty batch: nothing to do, nothing needed


def test_dispatch_rejects_shared_caches_and_bad_types(hyb):
    d = hyb.dims(4, 16, 10, 4, dtype=hyb.HYB_F32)
    f = 1 << 20
    meta = hyb.batch_meta(2, 2, seq_lens=f, block_tables=f, slot_mapping=f, state_slots=f, max_seq_len=32)
    a = hyb.layer_io(out=f, q=f, k=f, v=f, k_cache=f + 4096, v_cache=f + 8192)
    # two Full layers sharing one cache (the failure the vLLM page reports for shared caches)
    assert hyb.hyb_layer_dispatch([0, 0], 2, 0, [a, a], meta, d, 64, None, 0, 0) == hyb.HYB_ERR_INVALID_ARG
    # unknown layer type
    assert hyb.hyb_layer_dispatch([3], 1, 0, [a], meta, d, 64, None, 0, 0) == hyb.HYB_ERR_INVALID_ARG
    # decode with T != B
    meta_bad = hyb.batch_meta(2, 3, seq_lens=f, block_tables=f, slot_mapping=f, max_seq_len=32)
    assert hyb.hyb_layer_dispatch([0], 1, 0, [a], meta_bad, d, 64, None, 0, 0) == hyb.HYB_ERR_INVALID_ARG
    # Linear layer without a state pool
    lin = hyb.layer_io(out=f, q=f, k=f, v=f, num_state_slots=2)
    assert hyb.hyb_layer_dispatch([1], 1, 0, [lin], meta, d, 64, None, 0, 0) == hyb.HYB_ERR_INVALID_ARG
    # prefill mode: a Linear layer needs the chunked prefill's handoff workspace
    pmeta = hyb.batch_meta(2, 4, block_tables=f, slot_mapping=f, cu_q_lens=f, state_slots=f, max_q_len=2)
    linp = hyb.layer_io(out=f, q=f, k=f, v=f, state_pool=f + 4096, num_state_slots=2)
    assert hyb.hyb_layer_dispatch([1], 1, 1, [linp], pmeta, d, 64, None, 0, 0) == hyb.HYB_ERR_INVALID_ARG
    assert hyb.hyb_layer_dispatch([1], 1, 1, [linp], pmeta, d, 64, f + 8192, 64, 0) == hyb.HYB_ERR_INVALID_ARG
    # empty plan is a no-op
    assert hyb.hyb_layer_dispatch([], 0, 0, [], meta, d, 64, None, 0, 0) == hyb.HYB_OK


def test_sliding_window_arguments(hyb):
    f = 1 << 20
    d = hyb.dims(32, 128, 1000, 256)
    # a negative window is rejected by every Full-attention entry point
    dn = hyb.dims(32, 128, 1000, 256, window=-1)
    assert hyb.hyb_paged_kv_append(f, f, f, 4, f, f + 256, dn, 0) == hyb.HYB_ERR_INVALID_ARG
    assert hyb.hyb_paged_attn_decode(f, f, f, f, f, f, 2, 64, dn, f, 1 << 20, 0) == hyb.HYB_ERR_INVALID_ARG
    assert hyb.hyb_paged_attn_decode_noalloc(f, f, f, f, f, f, 2, 64, dn, 0) == hyb.HYB_ERR_INVALID_ARG
    assert hyb.hyb_paged_attn_prefill_causal(f, f, f, f, f, f, None, 2, 64, 32, dn, 0) == hyb.HYB_ERR_INVALID_ARG
    assert hyb.hyb_paged_attn_decode_workspace_size(2, 4096, dn) == 0
    # the decode workspace covers only the blocks a window can touch: (W + 14) // 16 + 1
    full = hyb.hyb_paged_attn_decode_workspace_size(8, 4096, d)
    w1000 = hyb.hyb_paged_attn_decode_workspace_size(8, 4096, hyb.dims(32, 128, 1000, 256, window=1000))
    w512 = hyb.hyb_paged_attn_decode_workspace_size(8, 4096, hyb.dims(32, 128, 1000, 256, window=512))
    w8k = hyb.hyb_paged_attn_decode_workspace_size(8, 4096, hyb.dims(32, 128, 1000, 256, window=8192))
    per_split = 8 * 32 * (128 * 4 + 8)
    assert full == 8 * per_split and w8k == full          # 256 blocks -> 8 splits of 32
    assert w1000 == 2 * per_split                         # 63 blocks -> 2 splits
    assert w512 == 2 * per_split                          # 33 blocks (unaligned start) -> 2
    assert hyb.hyb_paged_attn_decode_workspace_size(8, 4096, hyb.dims(32, 128, 1000, 256, window=497)) == 0


def test_dispatch_sliding_layer_arguments(hyb):
    d = hyb.dims(4, 16, 10, 4, dtype=hyb.HYB_F32)
    f = 1 << 20
    meta = hyb.batch_meta(2, 2, seq_lens=f, block_tables=f, slot_mapping=f, state_slots=f, max_seq_len=32)
    def io(window, off=0):
        return hyb.layer_io(out=f, q=f, k=f, v=f, k_cache=f + 4096 + off, v_cache=f + 8192 + off,
                            window=window)
    # a SLIDING layer needs a window > 0; FULL and LINEAR layers carry none
    assert hyb.hyb_layer_dispatch([2], 1, 0, [io(0)], meta, d, 64, None, 0, 0) == hyb.HYB_ERR_INVALID_ARG
    assert hyb.hyb_layer_dispatch([2], 1, 0, [io(-5)], meta, d, 64, None, 0, 0) == hyb.HYB_ERR_INVALID_ARG
    assert hyb.hyb_layer_dispatch([0], 1, 0, [io(8)], meta, d, 64, None, 0, 0) == hyb.HYB_ERR_INVALID_ARG
    # the dims' own window must be 0: windows come from the layer types
    dw = hyb.dims(4, 16, 10, 4, dtype=hyb.HYB_F32, window=8)
    assert hyb.hyb_layer_dispatch([2], 1, 0, [io(8)], meta, dw, 64, None, 0, 0) == hyb.HYB_ERR_INVALID_ARG
    # a SLIDING layer shares no cache with a FULL one
    assert hyb.hyb_layer_dispatch([0, 2], 2, 0, [io(0), io(8)], meta, d, 64, None, 0, 0) == hyb.HYB_ERR_INVALID_ARG


def test_lowp_state_step_arguments(hyb):
    f = 1 << 20
    # state dtype must be bf16 or fp16
    for bad in (hyb.HYB_F32, 7):
        assert hyb.hyb_linear_attn_step_lowp(f, f, f, f, f, bad, 4, f, 2, 4, 128, hyb.HYB_BF16, 0) == hyb.HYB_ERR_INVALID_ARG
    # a 16-bit pool is read in 16-byte pieces (8 columns): 16-byte alignment
    assert hyb.hyb_linear_attn_step_lowp(f, f, f, f, f + 4, hyb.HYB_F16, 4, f, 2, 4, 128, hyb.HYB_BF16, 0) == hyb.HYB_ERR_INVALID_ARG
    assert hyb.hyb_linear_attn_step_lowp(f, f, f, f, f + 8, hyb.HYB_F16, 4, f, 2, 4, 128, hyb.HYB_BF16, 0) == hyb.HYB_ERR_INVALID_ARG
    # no slots, unsupported head dim
    assert hyb.hyb_linear_attn_step_lowp(f, f, f, f, f, hyb.HYB_BF16, 0, f, 2, 4, 128, hyb.HYB_BF16, 0) == hyb.HYB_ERR_INVALID_ARG
    assert hyb.hyb_linear_attn_step_lowp(f, f, f, f, f, hyb.HYB_BF16, 4, f, 2, 4, 48, hyb.HYB_BF16, 0) == hyb.HYB_ERR_UNSUPPORTED
    # B = 0 is a no-op
    assert hyb.hyb_linear_attn_step_lowp(None, None, None, None, None, hyb.HYB_BF16, 4, None, 0, 4, 128, hyb.HYB_BF16, 0) == hyb.HYB_OK


def test_trace_without_a_traced_dispatch(hyb):
    """No dispatch has been traced on this thread: nothing to report (no CUDA call made)."""
    st, _ = hyb.hyb_trace_layer_ms(4)
    assert st == hyb.HYB_ERR_INVALID_ARG


def test_selftest_limit_checked_before_launch(hyb):
    """The bounded-wait self-test rejects a limit outside [1 us, 1 s] before any CUDA call."""
    assert hyb.hyb_selftest_bounded_waits(0, 0) == hyb.HYB_ERR_INVALID_ARG
    assert hyb.hyb_selftest_bounded_waits(1000001, 0) == hyb.HYB_ERR_INVALID_ARG


def test_noalloc_decode_checks_arguments_like_the_workspace_decode(hyb):
    """The allocation-free decode runs the workspace decode's own argument checks before
    any CUDA call (this container has no GPU): same status for the same bad arguments."""
    f = 1 << 20
    d = hyb.dims(32, 128, 1000, 256)
    cases = [
        (f, f, f, f, f, f, 2, 64, None),                          # no dims
        (None, f, f, f, f, f, 2, 64, d),                          # null output
        (f + 2, f, f, f, f, f, 2, 64, d),                         # misaligned output
        (f, f, f, f, f + 1, f, 2, 64, d),                         # misaligned block table
        (f, f, f, f, f, f, -1, 64, d),                            # negative batch
        (f, f, f, f, f, f, 2, 256 * 16 + 1, d),                   # beyond the block table
        (f, f, f, f, f, f, 2, 64, hyb.dims(32, 96, 1000, 256)),   # head dim without a kernel
        (f, f, f, f, f, f, 2, 64, hyb.dims(32, 128, 1000, 256, block_size=24)),
    ]
    for a in cases:
        want = hyb.hyb_paged_attn_decode(*a, f, 1 << 24, 0)
        assert want != hyb.HYB_OK
        assert hyb.hyb_paged_attn_decode_noalloc(*a, 0) == want, a
    # an empty batch is accepted before any pointer is looked at, and launches nothing
    assert hyb.hyb_paged_attn_decode_noalloc(None, None, None, None, None, None, 0, 0, d, 0) == hyb.HYB_OK
