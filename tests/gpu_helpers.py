"""Shared helpers of the GPU parity tests: host <-> device copies of the seeded inputs,
and the tolerance rules the tests apply.

Tolerances (floating point): bf16/fp32 attention outputs pass when every element has
|gpu - ref| <= 2e-2 + 1e-2 * |ref| (the allclose reading of "2e-2 max-abs / 1e-2
relative"); fp32
linear states pass when, for every (request, head) matrix, max|gpu - ref| <=
1e-3 * max|ref|. Integer and byte results (slots, cache images) must be identical.
"""
import numpy as np
import torch

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


def poisoned_pool(num_blocks, H, D, dtype_code):
    shape = (num_blocks, H, W.BLOCK_SIZE, D)
    if dtype_code == W.BF16:
        return np.full(shape, 0x7FC0, np.uint16)
    return np.full(shape, np.nan, np.float32)
