"""Blocks of 32 and 64 tokens (the vLLM/SGLang page uses 32) through the C ABI: slot
mapping, append, paged decode, tensor-core and CUDA-core prefill, with and without a
sliding window and released blocks, against the oracle at the same block size."""
import numpy as np
import pytest

import workloads as W
from gpu_helpers import (PagedCase, assert_out_close, decode_case, decode_gpu, released,
                         same_bytes, to_host)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("bs", [32, 64])
@pytest.mark.parametrize("dtype,H,D", [(W.BF16, 8, 128), (W.F32, 4, 64)])
def test_decode_larger_blocks(hyb, devstatus, bs, dtype, H, D):
    lens = [1, 31, 32, 33, 64, 65, 513, 2000, 4096]
    c = decode_case(600 + bs + D, lens, H, D, dtype, bs)
    out, _ = decode_gpu(hyb, c, 0, c.pool.block_tables)
    assert_out_close(out, c.decode_ref(), f"decode bs={bs}")
    outw, _ = decode_gpu(hyb, c, 100, released(c.pool.block_tables, c.ctx, 100, bs))
    assert_out_close(outw, c.decode_ref(100), f"decode bs={bs} W=100")
    assert devstatus() == (0, 0)


def test_decode_block_32_single_layer_workload(hyb, devstatus):
    """32 requests, lengths 128..4096, H=32, D=128, in 32-token blocks: every output."""
    db = W.decode_single_layer(0)
    c = decode_case(620, db.seq_lens, db.H, db.D, W.BF16, 32)
    out, _ = decode_gpu(hyb, c, 0, c.pool.block_tables)
    assert_out_close(out, c.decode_ref(), "decode bs=32, 32 requests")
    assert devstatus() == (0, 0)


@pytest.mark.parametrize("bs", [32, 64])
@pytest.mark.parametrize("window", [0, 100])
@pytest.mark.parametrize("qlens,ctx", [
    ([1, 5, 127, 128, 129, 300], [0] * 6),
    ([77, 256, 1, 130], [16, 300, 511, 5]),
])
def test_prefill_tensor_core_larger_blocks(hyb, devstatus, bs, window, qlens, ctx):
    c = PagedCase(630 + bs + window + len(qlens), qlens, ctx, 4, 128, W.BF16, bs)
    bt = released(c.pool.block_tables, c.ctx, window, bs) if window else c.pool.block_tables
    out, slot, kc = c.prefill_gpu(hyb, window, bt)
    assert np.array_equal(slot, c.sm) and same_bytes(kc, c.okc)
    assert_out_close(out, c.prefill_ref(window), f"prefill bs={bs} W={window}")
    assert devstatus() == (0, 0)


@pytest.mark.parametrize("window", [0, 200])
def test_cuda_core_prefill_block_32(hyb, devstatus, window):
    """fp32, D=64 (no tensor-core kernel), contexts past 512 keys, 32-token blocks."""
    c = PagedCase(650 + window, [40, 3, 600], [700, 1030, 0], 4, 64, W.F32, 32)
    bt = released(c.pool.block_tables, c.ctx, window, 32) if window else c.pool.block_tables
    out, slot, _ = c.prefill_gpu(hyb, window, bt)
    assert np.array_equal(slot, c.sm)
    assert_out_close(out, c.prefill_ref(window), f"cuda-core prefill bs=32 W={window}")
    assert devstatus() == (0, 0)
