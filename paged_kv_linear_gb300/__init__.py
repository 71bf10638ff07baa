"""paged_kv_linear_gb300 -- Python binding of libhyb.so (argument marshalling only).

Every function here has the name and argument order of the C entry point declared in
include/hyb.h and does nothing but turn torch tensors / ints into pointers and call it;
all computation runs in the library's CUDA kernels. PyTorch supplies device memory and
streams. Importing builds libhyb.so in-tree when it is missing or older than its sources;
there is no fallback: if it cannot be built or loaded, importing the binding raises.

Device arguments accept CUDA torch tensors (contiguous) or raw integer addresses;
``stream`` accepts None (torch's current stream), a torch.cuda.Stream or a raw handle.
Each call returns the hyb_status_t code (0 = HYB_OK); ``check()`` raises on non-zero.
"""
from __future__ import annotations

import ctypes as C

from ._build import LIB, build  # noqa: F401  (build() compiles libhyb.so in-tree)

HYB_OK, HYB_ERR_INVALID_ARG, HYB_ERR_UNSUPPORTED, HYB_ERR_CUDA, HYB_ERR_DEVICE_CHECK = range(5)
HYB_F32, HYB_BF16, HYB_F16 = 0, 1, 2
HYB_FULL, HYB_LINEAR, HYB_SLIDING = 0, 1, 2
HYB_MODE_DECODE, HYB_MODE_PREFILL = 0, 1
HYB_DEVERR_BAD_BLOCK, HYB_DEVERR_BAD_SLOT, HYB_DEVERR_BAD_STATE = 0x1, 0x2, 0x4
HYB_DEVERR_TIMEOUT, HYB_DEVERR_MISALIGNED, HYB_DEVERR_BAD_LENGTH = 0x8, 0x10, 0x20
BLOCK_SIZE = 16


class hyb_attn_dims_t(C.Structure):
    _fields_ = [("num_heads", C.c_int32), ("head_dim", C.c_int32), ("block_size", C.c_int32),
                ("num_blocks", C.c_int32), ("max_blocks_per_seq", C.c_int32),
                ("dtype", C.c_int32), ("scale", C.c_float), ("window", C.c_int32)]


class hyb_layer_io_t(C.Structure):
    _fields_ = [("out", C.c_void_p), ("q", C.c_void_p), ("k", C.c_void_p), ("v", C.c_void_p),
                ("k_cache", C.c_void_p), ("v_cache", C.c_void_p), ("state_pool", C.c_void_p),
                ("num_state_slots", C.c_int32), ("window", C.c_int32)]


class hyb_batch_meta_t(C.Structure):
    _fields_ = [("seq_lens", C.c_void_p), ("block_tables", C.c_void_p),
                ("slot_mapping", C.c_void_p), ("cu_q_lens", C.c_void_p),
                ("ctx_lens", C.c_void_p), ("state_slots", C.c_void_p), ("reset", C.c_void_p),
                ("B", C.c_int32), ("T", C.c_int32), ("max_seq_len", C.c_int32),
                ("max_q_len", C.c_int32)]


class HybError(RuntimeError):
    pass


def _load():
    from . import _build
    if _build.stale():
        try:
            _build.build()          # compile in-tree (nvcc, sm_103a) on first import
        except Exception as e:      # no toolkit / compile error: there is no other path
            raise ImportError(f"libhyb.so is missing or stale and could not be built: {e}") from e
    L = C.CDLL(LIB)
    p, i32, i64, u64, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_uint64, C.c_size_t
    sig = {
        "hyb_slot_mapping": [p, p, p, p, i32, i32, p, p],
        "hyb_paged_kv_append": [p, p, p, i32, p, p, p, p],
        "hyb_paged_attn_decode_workspace_size": ([i32, i32, p], sz),
        "hyb_paged_attn_decode": [p, p, p, p, p, p, i32, i32, p, p, sz, p],
        "hyb_paged_attn_decode_noalloc": [p, p, p, p, p, p, i32, i32, p, p],
        "hyb_paged_attn_decode_append": [p, p, p, p, p, p, p, p, p, i32, i32, p, p, sz, p],
        "hyb_paged_attn_prefill_causal": [p, p, p, p, p, p, p, i32, i32, i32, p, p],
        "hyb_linear_attn_step": [p, p, p, p, p, i32, p, i32, i32, i32, i32, p],
        "hyb_linear_attn_step_lowp": [p, p, p, p, p, i32, i32, p, i32, i32, i32, i32, p],
        "hyb_linear_attn_chunked_prefill": [p, p, p, p, p, p, p, i32, p, p, i32, i32, i32, i32,
                                            i32, i32, i32, p, sz, p],
        "hyb_linear_attn_chunked_prefill_workspace_size": ([], sz),
        "hyb_layer_dispatch": [p, i32, i32, p, p, p, i32, p, sz, p],
        "hyb_cache_bytes": ([i32, i32, i32, i32, i64, i32, i32, i32, p, p], u64),
        "hyb_device_status": [p, i32],
        "hyb_status_string": ([i32], C.c_char_p),
        "hyb_last_cuda_error": ([], C.c_char_p),
        "hyb_launch_count": ([i32], u64),
        "hyb_trace_layer_ms": [p, i32],
        "hyb_selftest_bounded_waits": [C.c_uint32, p],
    }
    for name, s in sig.items():
        fn = getattr(L, name)
        if isinstance(s, tuple):
            fn.argtypes, fn.restype = s
        else:
            fn.argtypes, fn.restype = s, i32
    return L


_lib = _load()


def lib():
    return _lib


# ------------------------------------------------------------------ marshalling
def _p(x):
    """Device pointer of a CUDA tensor (or a raw int / None)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_cuda:
        raise HybError("device argument is not a CUDA tensor")
    if not x.is_contiguous():
        raise HybError("device argument must be contiguous")
    return x.data_ptr()


def _d(d):
    """Pointer to a hyb_attn_dims_t (None passes NULL)."""
    return None if d is None else C.byref(d)


def _s(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def dtype_code(torch_dtype) -> int:
    import torch
    if torch_dtype == torch.bfloat16:
        return HYB_BF16
    if torch_dtype == torch.float32:
        return HYB_F32
    raise HybError(f"unsupported element type {torch_dtype}")


def dims(num_heads, head_dim, num_blocks, max_blocks_per_seq, dtype=HYB_BF16, scale=None,
         block_size=BLOCK_SIZE, window=0) -> hyb_attn_dims_t:
    if not isinstance(dtype, int):
        dtype = dtype_code(dtype)
    if scale is None:
        scale = head_dim ** -0.5
    return hyb_attn_dims_t(num_heads, head_dim, block_size, num_blocks, max_blocks_per_seq,
                           dtype, scale, window)


def check(status: int, what: str = "hyb call") -> None:
    if status != HYB_OK:
        extra = f" [{hyb_last_cuda_error()}]" if status == HYB_ERR_CUDA else ""
        raise HybError(f"{what}: {status_string(status)} (status {status}){extra}")


def hyb_last_cuda_error() -> str:
    return _lib.hyb_last_cuda_error().decode()


def status_string(status: int) -> str:
    return _lib.hyb_status_string(int(status)).decode()


# ------------------------------------------------------------------ entry points
def hyb_slot_mapping(slot_mapping, block_tables, cu_q_lens, ctx_lens, B, T, d, stream=None):
    return _lib.hyb_slot_mapping(_p(slot_mapping), _p(block_tables), _p(cu_q_lens), _p(ctx_lens),
                                 B, T, _d(d), _s(stream))


def hyb_paged_kv_append(k, v, slot_mapping, T, k_cache, v_cache, d, stream=None):
    return _lib.hyb_paged_kv_append(_p(k), _p(v), _p(slot_mapping), T, _p(k_cache), _p(v_cache),
                                    _d(d), _s(stream))


def hyb_paged_attn_decode_workspace_size(B, max_seq_len, d) -> int:
    return int(_lib.hyb_paged_attn_decode_workspace_size(B, max_seq_len, _d(d)))


def hyb_paged_attn_decode(out, q, k_cache, v_cache, block_tables, seq_lens, B, max_seq_len, d,
                          workspace, ws_bytes, stream=None):
    return _lib.hyb_paged_attn_decode(_p(out), _p(q), _p(k_cache), _p(v_cache), _p(block_tables),
                                      _p(seq_lens), B, max_seq_len, _d(d), _p(workspace),
                                      ws_bytes, _s(stream))


def hyb_paged_attn_decode_append(out, q, k, v, slot_mapping, k_cache, v_cache, block_tables,
                                 seq_lens, B, max_seq_len, d, workspace, ws_bytes, stream=None):
    return _lib.hyb_paged_attn_decode_append(_p(out), _p(q), _p(k), _p(v), _p(slot_mapping),
                                             _p(k_cache), _p(v_cache), _p(block_tables),
                                             _p(seq_lens), B, max_seq_len, _d(d),
                                             _p(workspace), ws_bytes, _s(stream))


def hyb_paged_attn_decode_noalloc(out, q, k_cache, v_cache, block_tables, seq_lens, B,
                                  max_seq_len, d, stream=None):
    """Paged decode whose split-K partials live in the library's own 16 MiB device array
    (for callers that cannot allocate device memory); see include/hyb.h."""
    return _lib.hyb_paged_attn_decode_noalloc(_p(out), _p(q), _p(k_cache), _p(v_cache),
                                              _p(block_tables), _p(seq_lens), B, max_seq_len,
                                              _d(d), _s(stream))


def hyb_paged_attn_prefill_causal(out, q, k_cache, v_cache, block_tables, cu_q_lens, ctx_lens,
                                  B, T, max_q_len, d, stream=None):
    return _lib.hyb_paged_attn_prefill_causal(_p(out), _p(q), _p(k_cache), _p(v_cache),
                                              _p(block_tables), _p(cu_q_lens), _p(ctx_lens), B,
                                              T, max_q_len, _d(d), _s(stream))


def hyb_linear_attn_step(out, q, k, v, state_pool, num_state_slots, state_slots, B, H, D, dtype,
                         stream=None):
    return _lib.hyb_linear_attn_step(_p(out), _p(q), _p(k), _p(v), _p(state_pool),
                                     num_state_slots, _p(state_slots), B, H, D, dtype,
                                     _s(stream))


def hyb_linear_attn_step_lowp(out, q, k, v, state_pool, state_dtype, num_state_slots, state_slots, B, H,
                              D, dtype, stream=None):
    """Linear step over a 16-bit (HYB_BF16 / HYB_F16) state pool, for the state-precision
    comparison; see include/hyb.h."""
    return _lib.hyb_linear_attn_step_lowp(_p(out), _p(q), _p(k), _p(v), _p(state_pool), state_dtype,
                                          num_state_slots, _p(state_slots), B, H, D, dtype, _s(stream))


def hyb_linear_attn_chunked_prefill(out, q, k, v, cu_seqlens, ctx_lens, state_pool,
                                    num_state_slots, state_slots, reset, B, T, max_len, H, D,
                                    chunk_size, dtype, workspace, ws_bytes, stream=None):
    return _lib.hyb_linear_attn_chunked_prefill(
        _p(out), _p(q), _p(k), _p(v), _p(cu_seqlens), _p(ctx_lens), _p(state_pool),
        num_state_slots, _p(state_slots), _p(reset), B, T, max_len, H, D, chunk_size, dtype,
        _p(workspace), ws_bytes, _s(stream))


def hyb_linear_attn_chunked_prefill_workspace_size() -> int:
    return int(_lib.hyb_linear_attn_chunked_prefill_workspace_size())


def layer_io(out=None, q=None, k=None, v=None, k_cache=None, v_cache=None, state_pool=None,
             num_state_slots=0, window=0) -> hyb_layer_io_t:
    return hyb_layer_io_t(_p(out), _p(q), _p(k), _p(v), _p(k_cache), _p(v_cache),
                          _p(state_pool), num_state_slots, window)


def batch_meta(B, T, seq_lens=None, block_tables=None, slot_mapping=None, cu_q_lens=None,
               ctx_lens=None, state_slots=None, reset=None, max_seq_len=0,
               max_q_len=0) -> hyb_batch_meta_t:
    return hyb_batch_meta_t(_p(seq_lens), _p(block_tables), _p(slot_mapping), _p(cu_q_lens),
                            _p(ctx_lens), _p(state_slots), _p(reset), B, T, max_seq_len,
                            max_q_len)


def hyb_layer_dispatch(layer_types, L, mode, layers, meta, d, chunk_size, workspace, ws_bytes,
                       stream=None):
    """layer_types: host sequence of ints; layers: sequence of hyb_layer_io_t (host);
    meta: hyb_batch_meta_t (host struct of device pointers)."""
    lt = (C.c_int32 * max(L, 1))(*[int(x) for x in layer_types])
    io = (hyb_layer_io_t * max(L, 1))(*layers)
    return _lib.hyb_layer_dispatch(lt, L, mode, io, C.byref(meta), _d(d), chunk_size,
                                   _p(workspace), ws_bytes, _s(stream))


def hyb_cache_bytes(L_full, L_linear, H, D, tokens, batch, kv_elem_bytes, state_elem_bytes):
    """Returns (total, full, linear) bytes."""
    full, lin = C.c_uint64(), C.c_uint64()
    tot = _lib.hyb_cache_bytes(L_full, L_linear, H, D, tokens, batch, kv_elem_bytes,
                               state_elem_bytes, C.byref(full), C.byref(lin))
    return int(tot), int(full.value), int(lin.value)


def hyb_device_status(clear: bool = True):
    """Returns (status, flags)."""
    flags = C.c_uint32()
    st = _lib.hyb_device_status(C.byref(flags), 1 if clear else 0)
    return int(st), int(flags.value)


def hyb_trace_layer_ms(L: int):
    """Per-layer device times (ms) of this thread's last dispatch traced with HYB_TRACE set;
    returns (status, list of L floats)."""
    buf = (C.c_float * max(L, 1))()
    st = _lib.hyb_trace_layer_ms(buf, L)
    return int(st), [float(x) for x in buf[:L]]


def hyb_selftest_bounded_waits(limit_us: int, stream=None):
    """Runs the bounded-wait self-test kernel: two waits nothing satisfies, each giving up
    after limit_us and setting HYB_DEVERR_TIMEOUT in the device status word."""
    return _lib.hyb_selftest_bounded_waits(limit_us, _s(stream))


def hyb_launch_count(reset: bool = False) -> int:
    return int(_lib.hyb_launch_count(1 if reset else 0))
