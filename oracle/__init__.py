"""CPU oracle for the hybrid-attention hot path (fp64, plain loops in C).

TEST INFRASTRUCTURE: only the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg import this package. The CUDA path never does, and
this package never imports the CUDA package.

``build()`` compiles ``oracle.c`` into ``liboracle.so`` next to it with gcc
(-O2, -ffp-contract=off, OpenMP when the compiler has it). The wrappers take
numpy arrays and return fp64 numpy arrays.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

BLOCK_SIZE = 16


def build(force: bool = False) -> str:
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = C.CDLL(_LIB)
            p, i32, i64, f64 = C.c_void_p, C.c_int, C.c_int64, C.c_double
            L.oracle_set_threads.argtypes = [i32]
            L.oracle_set_threads.restype = i32
            L.oracle_slot_mapping.argtypes = [p, i32, p, p, i32, i32, p]
            L.oracle_slot_mapping.restype = i32
            L.oracle_kv_append.argtypes = [p, p, p, i32, i32, i32, i32, i32, p, p]
            L.oracle_kv_append.restype = None
            L.oracle_full_decode.argtypes = [p, p, p, p, i32, p, i32, i32, i32, i32, i32, f64, i32, p]
            L.oracle_full_decode.restype = None
            L.oracle_full_prefill.argtypes = [p, p, p, p, i32, p, p, i32, i32, i32, i32, i32, f64, i32, p, i32, p]
            L.oracle_full_prefill.restype = None
            L.oracle_linear_recurrence.argtypes = [p, p, p, p, i32, i32, i32, i32, p, p, p, p, p]
            L.oracle_linear_recurrence.restype = None
            L.oracle_linear_recurrence_lowp.argtypes = [p, p, p, p, i32, i32, i32, i32, i32, p, p, p, p, p]
            L.oracle_linear_recurrence_lowp.restype = None
            L.oracle_linear_chunked.argtypes = [p, p, p, p, p, i32, i32, i32, i32, i32, p, p, p, p, p]
            L.oracle_linear_chunked.restype = None
            L.oracle_cache_bytes.argtypes = [i32, i32, i32, i32, i64, i32, i32, i32, p, p]
            L.oracle_cache_bytes.restype = C.c_uint64
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dt):
    return None if a is None else np.ascontiguousarray(a, dtype=dt)


def _elem(a):
    """(contiguous array, dtype code): uint16 arrays are bf16 bit patterns, float32 is fp32."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return a, 1
    if a.dtype == np.float32:
        return a, 0
    raise TypeError(f"oracle inputs are bf16 bit patterns (uint16) or float32, got {a.dtype}")


def set_threads(n: int = 0) -> int:
    """Set the OpenMP thread count (0 keeps the current one); returns the count in use."""
    return int(lib().oracle_set_threads(int(n)))


def slot_mapping(block_tables, cu_q_lens, ctx_lens=None, block_size=BLOCK_SIZE):
    bt = _c(block_tables, np.int32)
    cu = _c(cu_q_lens, np.int32)
    B = len(cu) - 1
    out = np.empty(int(cu[-1]), dtype=np.int64)
    rc = lib().oracle_slot_mapping(_ptr(bt), bt.shape[1], _ptr(cu), _ptr(_c(ctx_lens, np.int32)),
                                   B, block_size, _ptr(out))
    if rc != 0:
        raise ValueError("a position needs a logical block beyond the block table")
    return out


def kv_append(k, v, slot_map, k_cache, v_cache, block_size=BLOCK_SIZE):
    """Writes into k_cache / v_cache (numpy, [NB][H][bs][D]) in place."""
    k, dt = _elem(k)
    v, _ = _elem(v)
    T, H, D = k.shape
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous and k_cache.dtype == k.dtype
    sm = _c(slot_map, np.int64)
    lib().oracle_kv_append(_ptr(k), _ptr(v), _ptr(sm), T, H, D, block_size, k.itemsize,
                           _ptr(k_cache), _ptr(v_cache))


def full_decode(q, k_cache, v_cache, block_tables, seq_lens, scale, block_size=BLOCK_SIZE, window=0):
    q, dt = _elem(q)
    B, H, D = q.shape
    kc, _ = _elem(k_cache)
    vc, _ = _elem(v_cache)
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    out = np.zeros((B, H, D), dtype=np.float64)
    lib().oracle_full_decode(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(sl), B, H, D,
                             block_size, dt, float(scale), int(window), _ptr(out))
    return out


def full_prefill(q, k_cache, v_cache, block_tables, cu_q_lens, ctx_lens, scale, rows=None,
                 block_size=BLOCK_SIZE, window=0):
    q, dt = _elem(q)
    T, H, D = q.shape
    kc, _ = _elem(k_cache)
    vc, _ = _elem(v_cache)
    bt = _c(block_tables, np.int32)
    cu = _c(cu_q_lens, np.int32)
    B = len(cu) - 1
    r = _c(rows, np.int32)
    n = T if r is None else len(r)
    out = np.zeros((n, H, D), dtype=np.float64)
    lib().oracle_full_prefill(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(cu),
                              _ptr(_c(ctx_lens, np.int32)), B, H, D, block_size, dt, float(scale),
                              int(window), _ptr(r), 0 if r is None else len(r), _ptr(out))
    return out


def linear_recurrence(q, k, v, cu_seqlens, state_pool=None, state_slots=None, reset=None):
    q, dt = _elem(q)
    k, _ = _elem(k)
    v, _ = _elem(v)
    T, H, D = q.shape
    cu = _c(cu_seqlens, np.int32)
    B = len(cu) - 1
    out = np.zeros((T, H, D), dtype=np.float64)
    st = np.zeros((B, H, D, D), dtype=np.float64)
    lib().oracle_linear_recurrence(_ptr(q), _ptr(k), _ptr(v), _ptr(cu), B, H, D, dt,
                                   _ptr(_c(state_pool, np.float32)), _ptr(_c(state_slots, np.int32)),
                                   _ptr(_c(reset, np.uint8)), _ptr(out), _ptr(st))
    return out, st


def linear_recurrence_lowp(q, k, v, cu_seqlens, state_dtype, state_pool=None, state_slots=None,
                           reset=None):
    """The recurrence with a 16-bit state (state_dtype 1 = bf16, 2 = fp16): returns
    (out fp64 [T][H][D], final states as uint16 bit patterns [B][H][D][D])."""
    q, dt = _elem(q)
    k, _ = _elem(k)
    v, _ = _elem(v)
    T, H, D = q.shape
    cu = _c(cu_seqlens, np.int32)
    B = len(cu) - 1
    out = np.zeros((T, H, D), dtype=np.float64)
    st = np.zeros((B, H, D, D), dtype=np.uint16)
    lib().oracle_linear_recurrence_lowp(_ptr(q), _ptr(k), _ptr(v), _ptr(cu), B, H, D, dt,
                                        int(state_dtype), _ptr(_c(state_pool, np.uint16)),
                                        _ptr(_c(state_slots, np.int32)), _ptr(_c(reset, np.uint8)),
                                        _ptr(out), _ptr(st))
    return out, st


def linear_chunked(q, k, v, cu_seqlens, chunk, ctx_lens=None, state_pool=None, state_slots=None,
                   reset=None):
    q, dt = _elem(q)
    k, _ = _elem(k)
    v, _ = _elem(v)
    T, H, D = q.shape
    cu = _c(cu_seqlens, np.int32)
    B = len(cu) - 1
    out = np.zeros((T, H, D), dtype=np.float64)
    st = np.zeros((B, H, D, D), dtype=np.float64)
    lib().oracle_linear_chunked(_ptr(q), _ptr(k), _ptr(v), _ptr(cu), _ptr(_c(ctx_lens, np.int32)),
                                B, H, D, int(chunk), dt, _ptr(_c(state_pool, np.float32)),
                                _ptr(_c(state_slots, np.int32)), _ptr(_c(reset, np.uint8)),
                                _ptr(out), _ptr(st))
    return out, st


def linear_step(q, k, v, state_pool, state_slots):
    """One decode token per request: the recurrence over a single row each.
    Returns (out fp64 [B][H][D], new states fp64 [B][H][D][D])."""
    B = q.shape[0]
    cu = np.arange(B + 1, dtype=np.int32)
    return linear_recurrence(q, k, v, cu, state_pool, state_slots, None)


def cache_bytes(L_full, L_linear, H, D, tokens, batch, kv_elem_bytes, state_elem_bytes):
    full = C.c_uint64()
    lin = C.c_uint64()
    tot = lib().oracle_cache_bytes(L_full, L_linear, H, D, tokens, batch, kv_elem_bytes,
                                   state_elem_bytes, C.byref(full), C.byref(lin))
    return int(tot), int(full.value), int(lin.value)
