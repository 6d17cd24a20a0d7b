"""CPU oracle for the paged GQA decode step — TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its
Python binding) never imports it, and this package imports nothing from the
product.  Arrays are numpy: bf16 data travels as ``uint16`` bit patterns,
f32 as ``float32``.

Functions and the passages they follow (page title, section):
  rope_tables     Llama example page, ``src/rope.linnet`` (``tables``)
  rope_write_kv   Llama example page, ``src/attention.linnet`` (``decode``:
                  rope on q and k, ``write_at`` of k and v), with the paged
                  slot of the llama-3.1-8b-instruct architecture page
                  (``decode_paged`` signature, ``PageSize = 64``)
  decode          Llama example page, ``src/attention.linnet`` (``decode``:
                  ``seen[s] = s <= pos``, ``rsqrt(f32(head dim))``,
                  ``grouped_attention``), window from the gpt-oss-20b page;
                  optional attention sinks (gpt-oss-20b page, SinkAttention
                  ``param sinks``) as one value-less logit per query head
  step            rope_write_kv followed by decode
  prefill_paged   packed prompt tokens: rope, write at their pool slots, then
                  each token's causal attention over its row (the
                  llama-3.1-8b-instruct page's ``prefill_paged`` signature)
  packed          Llama example page, ``src/attention.linnet`` (``packed``):
                  sequences packed into one row, mask ``own[i, j] =
                  segments[i] == segments[j] && positions[j] <= positions[i]``

Every function is pinned by tests under ``tests/test_oracle_*.py`` against
closed forms, brute force and invariants; the rotation direction of RoPE is
the one convention the pages leave unprinted (parity unpinned for the
direction alone).
"""
import ctypes
import os

import numpy as np

from . import build as _build

BF16 = 0
F32 = 1


class Shape(ctypes.Structure):
    _fields_ = [
        ("rows", ctypes.c_int32), ("heads", ctypes.c_int32), ("kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("pages_per_row", ctypes.c_int32), ("num_pages", ctypes.c_int32),
        ("dtype", ctypes.c_int32), ("window", ctypes.c_int32), ("rope_theta", ctypes.c_float),
    ]


_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        vp = ctypes.c_void_p
        L.oracle_rope_tables.argtypes = [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp]
        L.oracle_rope_write_kv.argtypes = [ctypes.POINTER(Shape)] + [vp] * 8
        L.oracle_decode.argtypes = [ctypes.POINTER(Shape)] + [vp] * 7
        L.oracle_decode_sinks.argtypes = [ctypes.POINTER(Shape)] + [vp] * 8
        L.oracle_step.argtypes = [ctypes.POINTER(Shape)] + [vp] * 10
        L.oracle_prefill_paged.argtypes = [ctypes.POINTER(Shape), ctypes.c_int] + [vp] * 13
        L.oracle_packed.argtypes = [ctypes.POINTER(Shape), ctypes.c_int] + [vp] * 10
        L.oracle_set_threads.argtypes = [ctypes.c_int]
        L.oracle_set_threads.restype = ctypes.c_int
        L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        L.oracle_f32_to_bf16.restype = ctypes.c_uint16
        for f in (L.oracle_rope_tables, L.oracle_rope_write_kv, L.oracle_decode, L.oracle_decode_sinks,
                  L.oracle_step, L.oracle_prefill_paged, L.oracle_packed):
            f.restype = ctypes.c_int
        _lib = L
    return _lib


def _np_dtype(dtype):
    return np.uint16 if dtype == BF16 else np.float32


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def make_shape(rows, heads, kv_heads, head_dim, pages_per_row, num_pages, dtype,
               window=0, rope_theta=0.0, page_size=64):
    return Shape(rows, heads, kv_heads, head_dim, page_size, pages_per_row, num_pages,
                 dtype, window, rope_theta)


def rope_tables(theta, head_dim, length, dtype):
    """cos, sin tables [length, head_dim] of T (uint16 bf16 bits or float32)."""
    t = _np_dtype(dtype)
    c = np.zeros((length, head_dim), dtype=t)
    s = np.zeros((length, head_dim), dtype=t)
    rc = lib().oracle_rope_tables(theta, head_dim, length, dtype, _ptr(c), _ptr(s))
    if rc != 0:
        raise ValueError(f"oracle_rope_tables status {rc}")
    return c, s


def rope_write_kv(shape, q, k_new, v_new, positions, table, k_pool, v_pool):
    """Returns q_out; k_pool and v_pool are updated in place.  Returns (q_out, status)."""
    q_out = np.empty_like(q)
    rc = lib().oracle_rope_write_kv(ctypes.byref(shape), _ptr(q), _ptr(k_new), _ptr(v_new),
                                    _ptr(positions), _ptr(table), _ptr(q_out), _ptr(k_pool),
                                    _ptr(v_pool))
    return q_out, rc


def decode(shape, q_rot, positions, table, k_pool, v_pool, sinks=None):
    """Returns (out in T, out in float64, status).  sinks: [Hq] of T or None."""
    out = np.zeros(q_rot.shape, dtype=q_rot.dtype)
    out64 = np.zeros(q_rot.shape, dtype=np.float64)
    rc = lib().oracle_decode_sinks(ctypes.byref(shape), _ptr(q_rot), _ptr(positions), _ptr(table),
                                   _ptr(k_pool), _ptr(v_pool), _ptr(sinks), _ptr(out), _ptr(out64))
    return out, out64, rc


def step(shape, q, k_new, v_new, positions, table, k_pool, v_pool):
    """Whole step; pools updated in place.  Returns (q_rot, out, out64, status)."""
    q_rot = np.empty_like(q)
    out = np.zeros(q.shape, dtype=q.dtype)
    out64 = np.zeros(q.shape, dtype=np.float64)
    rc = lib().oracle_step(ctypes.byref(shape), _ptr(q), _ptr(k_new), _ptr(v_new),
                           _ptr(positions), _ptr(table), _ptr(k_pool), _ptr(v_pool),
                           _ptr(q_rot), _ptr(out), _ptr(out64))
    return q_rot, out, out64, rc


def prefill_paged(shape, q, k_new, v_new, positions, rows, slots, table, k_pool, v_pool, sinks=None):
    """Prefill of packed tokens; pools updated in place.  Returns (q_rot, out, out64, status)."""
    q_rot = np.empty_like(q)
    out = np.zeros(q.shape, dtype=q.dtype)
    out64 = np.zeros(q.shape, dtype=np.float64)
    rc = lib().oracle_prefill_paged(ctypes.byref(shape), int(q.shape[0]), _ptr(q), _ptr(k_new), _ptr(v_new),
                                    _ptr(positions), _ptr(rows), _ptr(slots), _ptr(table), _ptr(k_pool),
                                    _ptr(v_pool), _ptr(sinks), _ptr(q_rot), _ptr(out), _ptr(out64))
    return q_rot, out, out64, rc


def packed(shape, q, k, v, positions, segments, sinks=None):
    """Packed attention; returns (q_rot, k_rot, out, out64, status)."""
    q_rot, k_rot = np.empty_like(q), np.empty_like(k)
    out = np.zeros(q.shape, dtype=q.dtype)
    out64 = np.zeros(q.shape, dtype=np.float64)
    rc = lib().oracle_packed(ctypes.byref(shape), int(q.shape[0]), _ptr(q), _ptr(k), _ptr(v), _ptr(positions),
                             _ptr(segments), _ptr(sinks), _ptr(q_rot), _ptr(k_rot), _ptr(out), _ptr(out64))
    return q_rot, k_rot, out, out64, rc


def set_threads(n: int) -> int:
    """Threads for the row loops (1 = serial); returns the count in use."""
    return int(lib().oracle_set_threads(int(n)))


def f32_to_bf16_bits(x: float) -> int:
    return int(lib().oracle_f32_to_bf16(float(x)))


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float32 (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)
