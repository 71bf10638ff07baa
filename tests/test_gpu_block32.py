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


@pytest.mark.parametrize("bs", [32, 64])
def test_decode_dispatch_larger_blocks(hyb, devstatus, bs):
    """A decode dispatch of [full, full, linear, full] layers over 32- / 64-token blocks, new
    rows placed through the block table: the Full layers after the first read their block
    ids and first tiles before waiting for the previous kernel. Each Full layer equals the
    oracle's append + decode on its own pool, and the Linear layer the oracle's step."""
    import torch
    import oracle
    from gpu_helpers import assert_states_close, empty_rows, to_dev
    lens = np.array([1, 31, 32, 33, 100, 700, 2049], np.int32)
    B, H, D = len(lens), 4, 128
    lt = [0, 0, 1, 0]
    g = W.rng(660 + bs)
    pool = W.block_pool(g, lens, block_size=bs)
    d = hyb.dims(H, D, pool.num_blocks, pool.max_blocks, W.BF16, block_size=bs)
    msl = int(lens.max())
    slots_h = g.permutation(B).astype(np.int32)
    host, ios, dev, outs = [], [], [], []
    for l, t in enumerate(lt):
        q, k, v = (W.rows(g, (B, H, D), D, W.BF16) for _ in range(3))
        out = empty_rows((B, H, D), W.BF16)
        x = [to_dev(q), to_dev(k), to_dev(v)]
        if t == 0:
            kc = W.rows(g, (pool.num_blocks, H, bs, D), D, W.BF16)
            vc = W.rows(g, (pool.num_blocks, H, bs, D), D, W.BF16)
            host.append((q, k, v, kc, vc))
            x += [to_dev(kc), to_dev(vc)]
            ios.append(hyb.layer_io(out, *x))
        else:
            st = W.synthetic_state(g, B, H, D, lens)
            host.append((q, k, v, st))
            x.append(to_dev(st))
            ios.append(hyb.layer_io(out, x[0], x[1], x[2], state_pool=x[3], num_state_slots=B))
        dev.append(x)
        outs.append(out)
    ws_n = hyb.hyb_paged_attn_decode_workspace_size(B, msl, d)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device="cuda")
    meta = hyb.batch_meta(B, B, seq_lens=to_dev(lens), block_tables=to_dev(pool.block_tables),
                          state_slots=to_dev(slots_h), max_seq_len=msl)
    hyb.check(hyb.hyb_layer_dispatch(lt, len(lt), 0, ios, meta, d, 64, ws, ws_n))
    torch.cuda.synchronize()
    sm = oracle.slot_mapping(pool.block_tables, np.arange(B + 1), lens - 1, block_size=bs)
    for l, t in enumerate(lt):
        if t == 0:
            q, k, v, kc, vc = host[l]
            oracle.kv_append(k, v, sm, kc, vc, block_size=bs)
            ref = oracle.full_decode(q, kc, vc, pool.block_tables, lens, D ** -0.5, block_size=bs)
            assert_out_close(outs[l], ref, f"layer {l} bs={bs}")
        else:
            q, k, v, st = host[l]
            o_ref, s_ref = oracle.linear_step(q, k, v, st, slots_h)
            assert_out_close(outs[l], o_ref, f"layer {l} (linear)")
            assert_states_close(to_host(dev[l][3])[slots_h], s_ref)
    assert devstatus() == (0, 0)
