"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This module only *draws* inputs: random q/k/v rows, sequence-length mixes, shuffled
block pools and block tables, synthetic linear states. It holds none of the
method's arithmetic (no slot mapping, no attention, no state update), so that
both sides of every parity check start from the same bytes while sharing no
compute code.

Shapes and distributions follow the hybrid-model pages:
  * Full-attention KV is paged in blocks of 16 tokens reached through a
    per-request block table ("推理框架适配Hybrid Model：KV Cache管理与算子调度实战", §2.1).
  * Request-length mix of 80% short / 20% long ("大模型混合架构推理优化：
    精度/稀疏/数据流/计算单元四维协同", §2.1).
Values: q, k, v ~ N(0, 1)/sqrt(D) drawn in fp32 and rounded once to bf16
(round-to-nearest-even) when the workload is bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 16

F32 = 0   # dtype codes used on both sides of the boundary
BF16 = 1


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


# ---------------------------------------------------------------- bf16 bytes
def bf16_round(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even; NaN -> quiet NaN."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    bias = 0x7FFF + ((u >> 16) & 1)
    r = ((u + bias) >> 16).astype(np.uint16)
    r[np.isnan(x)] = 0x7FC0
    return r


def bf16_to_f32(u: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp32 values (exact)."""
    u = np.ascontiguousarray(u, dtype=np.uint16)
    return (u.astype(np.uint32) << 16).view(np.float32)


def rows(g: np.random.Generator, shape, D: int, dtype: int) -> np.ndarray:
    """N(0,1)/sqrt(D) values; uint16 bf16 bit patterns for BF16, float32 for F32."""
    x = (g.standard_normal(size=shape, dtype=np.float32) / np.float32(math.sqrt(D))).astype(np.float32)
    return bf16_round(x) if dtype == BF16 else x


def unit_dirs(g: np.random.Generator, H: int, D: int) -> np.ndarray:
    """One random unit vector per head, fp32 [H][D]."""
    u = g.standard_normal(size=(H, D)).astype(np.float64)
    return (u / np.linalg.norm(u, axis=1, keepdims=True)).astype(np.float32)


def directed_rows(g: np.random.Generator, coef, u: np.ndarray, D: int, dtype: int,
                  noise: float = 1.0) -> np.ndarray:
    """Rows x[t][h] = coef[t][h] * u[h] + noise * N(0,1)/sqrt(D), drawn in fp32 and rounded
    once to bf16 for BF16. coef is [T] (same for every head) or [T][H]; u is [H][D].
    Gives inputs whose attention scores follow a chosen profile along the sequence
    (peaked or moving softmax maxima) while the values stay N(0,1)/sqrt(D)-like."""
    coef = np.asarray(coef, dtype=np.float32)
    if coef.ndim == 1:
        coef = coef[:, None]
    T, H = coef.shape[0], u.shape[0]
    x = g.standard_normal(size=(T, H, D), dtype=np.float32)
    x *= np.float32(noise / math.sqrt(D))
    x += coef[:, :, None] * u[None, :, :]
    return bf16_round(x) if dtype == BF16 else x


def esize(dtype: int) -> int:
    return 2 if dtype == BF16 else 4


def np_elem_dtype(dtype: int):
    return np.uint16 if dtype == BF16 else np.float32


# ------------------------------------------------------------- length mixes
def lens_uniform(g, B: int, lo: int, hi: int) -> np.ndarray:
    return g.integers(lo, hi + 1, size=B).astype(np.int32)


def lens_short_long(g, B: int, short_frac: float = 0.8, short_mu: float = 128.0,
                    long_mu: float = 2048.0, sigma: float = 0.5) -> np.ndarray:
    """80% ~ round(LogNormal(ln 128, 0.5)), 20% ~ round(LogNormal(ln 2048, 0.5)),
    clamped >= 1, then shuffled (sigma is not on the pages: 0.5 is a stated choice)."""
    n_short = int(round(B * short_frac))
    s = np.round(g.lognormal(math.log(short_mu), sigma, size=n_short))
    l = np.round(g.lognormal(math.log(long_mu), sigma, size=B - n_short))
    out = np.maximum(np.concatenate([s, l]), 1).astype(np.int32)
    g.shuffle(out)
    return out


# ---------------------------------------------------------- paged block pool
@dataclass
class BlockPool:
    num_blocks: int                 # NB physical blocks in the pool
    block_tables: np.ndarray        # int32 [B][MB]; -1 where a request owns no block
    blocks_per_req: np.ndarray      # int32 [B]
    used: np.ndarray                # int32 [n_used] physical ids handed out, in order

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])


def block_pool(g, capacity_tokens: np.ndarray, slack: float = 1.25, min_blocks: int = 0,
               block_size: int = BLOCK_SIZE) -> BlockPool:
    """Give request b ceil(capacity_tokens[b]/block_size) blocks drawn from a seeded
    Fisher-Yates shuffle of a pool of ceil(slack * total) blocks."""
    cap = np.asarray(capacity_tokens, dtype=np.int64)
    nb = (cap + block_size - 1) // block_size
    total = int(nb.sum())
    NB = max(int(math.ceil(slack * total)), min_blocks, 1)
    perm = g.permutation(NB).astype(np.int32)
    MB = max(int(nb.max()) if len(nb) else 1, 1)
    bt = np.full((len(cap), MB), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(nb):
        bt[b, :n] = perm[off:off + n]
        off += int(n)
    return BlockPool(NB, bt, nb.astype(np.int32), perm[:total].copy())


def synthetic_state(g, n: int, H: int, D: int, seq_lens: np.ndarray) -> np.ndarray:
    """fp32 [n][H][D][D] with entries ~ N(0, seq/D^2): the spread of a state after
    `seq` tokens of N(0,1/D) keys and values (used where a decode step has no prefill)."""
    st = g.standard_normal(size=(n, H, D, D), dtype=np.float32)
    sd = (np.sqrt(np.asarray(seq_lens, dtype=np.float64)) / D).astype(np.float32)
    st *= sd[:n, None, None, None]
    return st


def cu_from_lens(lens) -> np.ndarray:
    lens = np.asarray(lens, dtype=np.int64)
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


# ------------------------------------------------------------ named workloads
@dataclass
class DecodeBatch:
    """One decode token per request: Full layer appends then attends, Linear layer steps."""
    H: int
    D: int
    dtype: int
    seq_lens: np.ndarray            # int32 [B], includes the token appended this step
    pool: BlockPool
    extra: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return int(len(self.seq_lens))


def decode_single_layer(seed: int = 0, B: int = 32, H: int = 32, D: int = 128,
                        lo: int = 128, hi: int = 4096) -> DecodeBatch:
    """32 requests, seq_lens ~ U{128..4096}, blocks shuffled across a pool."""
    g = rng(seed)
    lens = lens_uniform(g, B, lo, hi)
    return DecodeBatch(H, D, BF16, lens, block_pool(g, lens))


def decode_hybrid_32layer(seed: int = 0, B: int = 64, H: int = 32, D: int = 128) -> DecodeBatch:
    """Batch of 64 with the 80%/20% short/long length mix, 32 layers [F,F,F,Lin]x8."""
    g = rng(seed)
    lens = lens_short_long(g, B)
    db = DecodeBatch(H, D, BF16, lens, block_pool(g, lens))
    db.extra["layer_types"] = np.array(([0, 0, 0, 1] * 8), dtype=np.int32)
    return db


def decode_long_context(seed: int = 0, B: int = 8, H: int = 32, D: int = 128,
                        ctx: int = 131072) -> DecodeBatch:
    """8 requests at 131072 tokens (8192 blocks each) placed at random in the pool."""
    g = rng(seed)
    lens = np.full(B, ctx, dtype=np.int32)
    return DecodeBatch(H, D, BF16, lens, block_pool(g, lens))


@dataclass
class PrefillBatch:
    H: int
    D: int
    dtype: int
    q_lens: np.ndarray              # int32 [B] tokens in this call
    ctx_lens: np.ndarray            # int32 [B] tokens already cached/accumulated before the call
    pool: BlockPool
    chunk: int = 64


def prefill_chunked(seed: int = 0, B: int = 8, L: int = 8192, H: int = 32, D: int = 128,
                    chunk: int = 64) -> PrefillBatch:
    """8 requests x 8192-token prompts; Full layer writes a shuffled paged pool."""
    g = rng(seed)
    lens = np.full(B, L, dtype=np.int32)
    return PrefillBatch(H, D, BF16, lens, np.zeros(B, np.int32), block_pool(g, lens), chunk)


def tiny_hybrid_pair(seed: int = 0):
    """H=2, D=16, fp32, prompts 5 and 37, 16-block pool as a seeded permutation,
    then 4 decode steps (final lengths 9 and 41)."""
    g = rng(seed)
    prompts = np.array([5, 37], dtype=np.int32)
    steps = 4
    final = prompts + steps
    pool = block_pool(g, final, slack=1.0, min_blocks=16)
    return dict(H=2, D=16, dtype=F32, prompts=prompts, steps=steps, pool=pool, g=g)


# --------------------------------------------------------- device-side fills
def device_rows_(t, seed: int, D: int):
    """Fill a torch tensor (bf16 or fp32, any device) with N(0,1)/sqrt(D), seeded.
    Used for multi-GB pools where drawing on the host would dominate set-up time;
    parity checks copy the sampled parts back to the host for the oracle."""
    import torch
    gen = torch.Generator(device=t.device)
    gen.manual_seed(seed)
    n = t.numel()
    flat = t.view(-1)
    step = 1 << 28
    for s in range(0, n, step):
        e = min(n, s + step)
        x = torch.randn(e - s, generator=gen, device=t.device, dtype=torch.float32)
        x.mul_(1.0 / math.sqrt(D))
        flat[s:e].copy_(x)
    return t


def device_state_(t, seed: int, seq_lens, D: int):
    """Fill an fp32 [n][H][D][D] state tensor with N(0, seq/D^2) entries, seeded."""
    import torch
    gen = torch.Generator(device=t.device)
    gen.manual_seed(seed)
    for i in range(t.shape[0]):
        x = torch.randn(t[i].shape, generator=gen, device=t.device, dtype=torch.float32)
        x.mul_(math.sqrt(float(seq_lens[i])) / D)
        t[i].copy_(x)
    return t
