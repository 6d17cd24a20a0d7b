"""ctypes binding of libpdattn (include/pdattn.h).

Argument marshalling only: every function takes torch tensors that already
live on the GPU, checks their shapes and dtypes against the parameters, and
passes raw device pointers and the current CUDA stream to the C-ABI call of
the same name.  No computation happens here, and there is no fallback: if the
library is missing, importing this module raises.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpdattn.so")

OK, EINVAL, EUNSUPPORTED, ECUDA, EBADPAGE, ETIMEOUT, EBADPOS = range(7)
BF16, F32 = 0, 1
_DTYPES = {torch.bfloat16: BF16, torch.float32: F32}


class PdattnError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"pdattn status {status}: {msg}")
        self.status = status


class Params(ctypes.Structure):
    _fields_ = [
        ("rows", ctypes.c_int32), ("heads", ctypes.c_int32), ("kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("pages_per_row", ctypes.c_int32), ("num_pages", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("window", ctypes.c_int32), ("scale", ctypes.c_float), ("rope_cos", ctypes.c_void_p),
        ("rope_sin", ctypes.c_void_p), ("rope_len", ctypes.c_int32), ("chunk_pages", ctypes.c_int32),
        ("sinks", ctypes.c_void_p),
    ]


class Layer(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p),
        ("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p), ("out", ctypes.c_void_p),
        ("window", ctypes.c_int32), ("reserved", ctypes.c_int32), ("sinks", ctypes.c_void_p),
    ]


LAYERS_PER_LAUNCH = 32


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -m paged_gqa_decode_step_gb300.build` (nvcc, sm_103a)")
    L = ctypes.CDLL(LIB_PATH)
    vp, sz, i32, P = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.POINTER(Params)
    sig = {
        "pdattn_workspace_size": (sz, [P]),
        "pdattn_rope_tables": (i32, [ctypes.c_float, i32, i32, i32, vp, vp, vp]),
        "pdattn_rope_write_kv": (i32, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "pdattn_plan": (i32, [P, vp, vp, sz, vp]),
        "pdattn_attend": (i32, [P, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "pdattn_decode": (i32, [P, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "pdattn_decode_fused": (i32, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "pdattn_decode_fused_noalloc": (i32, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
        "pdattn_layers_workspace_size": (sz, [P, i32]),
        "pdattn_decode_layers": (i32, [P, i32, ctypes.POINTER(Layer), vp, vp, vp, sz, vp]),
        "pdattn_prefill_workspace_size": (sz, [P, i32]),
        "pdattn_prefill_paged": (i32, [P, i32] + [vp] * 11 + [sz, vp]),
        "pdattn_prefill_attend": (i32, [P, i32] + [vp] * 6 + [sz, vp]),
        "pdattn_packed_workspace_size": (sz, [P, i32]),
        "pdattn_packed": (i32, [P, i32] + [vp] * 7 + [sz, vp]),
        "pdattn_packed_attend": (i32, [P, i32] + [vp] * 4 + [sz, vp]),
        "pdattn_check_status": (i32, [vp, vp]),
        "pdattn_last_error": (ctypes.c_char_p, []),
        "pdattn_last_launch_count": (i32, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype, f.argtypes = res, args
    return L


lib = _load()


def _check(status):
    if status != OK:
        raise PdattnError(status, lib.pdattn_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def make_params(rows, heads, kv_heads, head_dim, pages_per_row, num_pages, dtype, window=0, scale=0.0,
                rope_cos=None, rope_sin=None, chunk_pages=0, sinks=None):
    """Parameter block; rope tables (torch tensors [len, D]) keep rotation on;
    sinks: optional [heads] tensor of the element type (attention sinks)."""
    p = Params(rows, heads, kv_heads, head_dim, 64, pages_per_row, num_pages, _DTYPES[dtype], window,
               scale, None, None, 0, chunk_pages, None)
    if sinks is not None:
        _expect("sinks", sinks, (heads,), dtype)
        p.sinks = sinks.data_ptr()
        p._sinks = sinks
    if rope_cos is not None:
        for name, t in (("rope_cos", rope_cos), ("rope_sin", rope_sin)):
            _expect(name, t, (rope_cos.shape[0], head_dim), dtype)
        p.rope_cos, p.rope_sin, p.rope_len = rope_cos.data_ptr(), rope_sin.data_ptr(), rope_cos.shape[0]
        # the block holds raw pointers: keep the tables alive as long as it lives
        p._tables = (rope_cos, rope_sin)
    return p


def workspace_size(p):
    n = lib.pdattn_workspace_size(ctypes.byref(p))
    if n == 0:
        raise PdattnError(EINVAL, lib.pdattn_last_error().decode())
    return n


def new_workspace(p, device="cuda"):
    """A zero-filled workspace of the right size (uint8 tensor, 256-byte aligned)."""
    return torch.zeros(workspace_size(p), dtype=torch.uint8, device=device)


def rope_tables(theta, head_dim, length, dtype, device="cuda", stream=None):
    cos = torch.empty(length, head_dim, dtype=dtype, device=device)
    sin = torch.empty(length, head_dim, dtype=dtype, device=device)
    _check(lib.pdattn_rope_tables(theta, head_dim, length, _DTYPES[dtype], _ptr(cos), _ptr(sin), _stream(stream)))
    return cos, sin


def _ws(ws):
    if not (ws.is_cuda and ws.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    return _ptr(ws), ws.numel() * ws.element_size()


def _expect(name, t, shape, dtype):
    """Shape, dtype, device and contiguity of one argument."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _dt(p):
    return torch.bfloat16 if p.dtype == BF16 else torch.float32


def _check_common(p, positions, table, k_pool, v_pool):
    _expect("positions", positions, (p.rows,), torch.int32)
    _expect("table", table, (p.rows, p.pages_per_row), torch.int32)
    pool = (p.num_pages, p.kv_heads, 64, p.head_dim)
    _expect("k_pool", k_pool, pool, _dt(p))
    _expect("v_pool", v_pool, pool, _dt(p))


def _check_q(p, **named):
    for name, t in named.items():
        h = p.heads if name in ("q", "q_rot", "q_out", "out") else p.kv_heads
        _expect(name, t, (p.rows, h, p.head_dim), _dt(p))


def rope_write_kv(p, q, k_new, v_new, positions, table, q_out, k_pool, v_pool, ws, stream=None):
    _check_common(p, positions, table, k_pool, v_pool)
    _check_q(p, q=q, k_new=k_new, v_new=v_new, q_out=q_out)
    w, n = _ws(ws)
    _check(lib.pdattn_rope_write_kv(ctypes.byref(p), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(positions),
                                    _ptr(table), _ptr(q_out), _ptr(k_pool), _ptr(v_pool), w, n, _stream(stream)))


def plan(p, positions, ws, stream=None):
    _expect("positions", positions, (p.rows,), torch.int32)
    w, n = _ws(ws)
    _check(lib.pdattn_plan(ctypes.byref(p), _ptr(positions), w, n, _stream(stream)))


def attend(p, q_rot, positions, table, k_pool, v_pool, out, ws, stream=None):
    _check_common(p, positions, table, k_pool, v_pool)
    _check_q(p, q_rot=q_rot, out=out)
    w, n = _ws(ws)
    _check(lib.pdattn_attend(ctypes.byref(p), _ptr(q_rot), _ptr(positions), _ptr(table), _ptr(k_pool),
                             _ptr(v_pool), _ptr(out), w, n, _stream(stream)))


def decode(p, q_rot, positions, table, k_pool, v_pool, out, ws, stream=None):
    _check_common(p, positions, table, k_pool, v_pool)
    _check_q(p, q_rot=q_rot, out=out)
    w, n = _ws(ws)
    _check(lib.pdattn_decode(ctypes.byref(p), _ptr(q_rot), _ptr(positions), _ptr(table), _ptr(k_pool),
                             _ptr(v_pool), _ptr(out), w, n, _stream(stream)))


def decode_fused(p, q, k_new, v_new, positions, table, k_pool, v_pool, out, ws, stream=None):
    _check_common(p, positions, table, k_pool, v_pool)
    _check_q(p, q=q, k_new=k_new, v_new=v_new, out=out)
    w, n = _ws(ws)
    _check(lib.pdattn_decode_fused(ctypes.byref(p), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(positions),
                                   _ptr(table), _ptr(k_pool), _ptr(v_pool), _ptr(out), w, n, _stream(stream)))


def decode_fused_noalloc(p, q, k_new, v_new, positions, table, k_pool, v_pool, out, stream=None):
    """decode_fused with the library's fixed scratch array instead of a workspace."""
    _check_common(p, positions, table, k_pool, v_pool)
    _check_q(p, q=q, k_new=k_new, v_new=v_new, out=out)
    _check(lib.pdattn_decode_fused_noalloc(ctypes.byref(p), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(positions),
                                           _ptr(table), _ptr(k_pool), _ptr(v_pool), _ptr(out), _stream(stream)))


def layers_workspace_size(p, n_layers):
    n = lib.pdattn_layers_workspace_size(ctypes.byref(p), n_layers)
    if n == 0:
        raise PdattnError(EINVAL, lib.pdattn_last_error().decode() or "invalid parameters")
    return n


def new_layers_workspace(p, n_layers, device="cuda"):
    return torch.zeros(layers_workspace_size(p, n_layers), dtype=torch.uint8, device=device)


def decode_layers(p, layers, positions, table, ws, stream=None):
    """The decode step of several layers in one group of launches (per 32 layers).
    layers: a sequence of dicts with q, k_new, v_new, k_pool, v_pool, out
    (tensors shaped as for decode_fused) and optional window (int) and sinks
    ([heads] tensor); p.window and p.sinks are not read."""
    _expect("positions", positions, (p.rows,), torch.int32)
    _expect("table", table, (p.rows, p.pages_per_row), torch.int32)
    arr = (Layer * max(1, len(layers)))()
    keep = []
    pool = (p.num_pages, p.kv_heads, 64, p.head_dim)
    for i, y in enumerate(layers):
        _check_q(p, q=y["q"], k_new=y["k_new"], v_new=y["v_new"], out=y["out"])
        _expect("k_pool", y["k_pool"], pool, _dt(p))
        _expect("v_pool", y["v_pool"], pool, _dt(p))
        sinks = y.get("sinks")
        if sinks is not None:
            _expect("sinks", sinks, (p.heads,), _dt(p))
        arr[i] = Layer(y["q"].data_ptr(), y["k_new"].data_ptr(), y["v_new"].data_ptr(), y["k_pool"].data_ptr(),
                       y["v_pool"].data_ptr(), y["out"].data_ptr(), int(y.get("window", 0)), 0,
                       None if sinks is None else sinks.data_ptr())
        keep.append(y)
    w, n = _ws(ws)
    _check(lib.pdattn_decode_layers(ctypes.byref(p), len(layers), arr, _ptr(positions), _ptr(table), w, n,
                                    _stream(stream)))


def prefill_workspace_size(p, n_tokens):
    n = lib.pdattn_prefill_workspace_size(ctypes.byref(p), n_tokens)
    if n == 0:
        raise PdattnError(EINVAL, lib.pdattn_last_error().decode() or "invalid parameters")
    return n


def new_prefill_workspace(p, n_tokens, device="cuda"):
    return torch.zeros(prefill_workspace_size(p, n_tokens), dtype=torch.uint8, device=device)


def prefill_paged(p, q, k_new, v_new, positions, rows, slots, table, k_pool, v_pool, out, ws, stream=None):
    """Packed prompt tokens: q / out [P, heads, D], k_new / v_new [P, kv_heads, D],
    positions / rows / slots [P] int32; p.rows is the number of table rows."""
    n = q.shape[0] if isinstance(q, torch.Tensor) else -1
    _expect("table", table, (p.rows, p.pages_per_row), torch.int32)
    pool = (p.num_pages, p.kv_heads, 64, p.head_dim)
    _expect("k_pool", k_pool, pool, _dt(p))
    _expect("v_pool", v_pool, pool, _dt(p))
    for name, t in (("positions", positions), ("rows", rows), ("slots", slots)):
        _expect(name, t, (n,), torch.int32)
    for name, t, h in (("q", q, p.heads), ("k_new", k_new, p.kv_heads), ("v_new", v_new, p.kv_heads),
                       ("out", out, p.heads)):
        _expect(name, t, (n, h, p.head_dim), _dt(p))
    w, nb = _ws(ws)
    _check(lib.pdattn_prefill_paged(ctypes.byref(p), n, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(positions),
                                    _ptr(rows), _ptr(slots), _ptr(table), _ptr(k_pool), _ptr(v_pool), _ptr(out),
                                    w, nb, _stream(stream)))


def prefill_attend(p, positions, table, k_pool, v_pool, out, ws, stream=None):
    """Attention half of prefill_paged, over what its last call left in ws."""
    n = out.shape[0] if isinstance(out, torch.Tensor) else -1
    _expect("positions", positions, (n,), torch.int32)
    _expect("table", table, (p.rows, p.pages_per_row), torch.int32)
    pool = (p.num_pages, p.kv_heads, 64, p.head_dim)
    _expect("k_pool", k_pool, pool, _dt(p))
    _expect("v_pool", v_pool, pool, _dt(p))
    _expect("out", out, (n, p.heads, p.head_dim), _dt(p))
    w, nb = _ws(ws)
    _check(lib.pdattn_prefill_attend(ctypes.byref(p), n, _ptr(positions), _ptr(table), _ptr(k_pool), _ptr(v_pool),
                                     _ptr(out), w, nb, _stream(stream)))


def new_packed_workspace(p, n_tokens, device="cuda"):
    n = lib.pdattn_packed_workspace_size(ctypes.byref(p), n_tokens)
    if n == 0:
        raise PdattnError(EINVAL, lib.pdattn_last_error().decode() or "invalid parameters")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def packed(p, q, k, v, positions, segments, out, ws, stream=None):
    """Sequences packed into one row: q / out [n, heads, D], k / v [n, kv_heads, D],
    positions / segments [n] int32."""
    n = q.shape[0] if isinstance(q, torch.Tensor) else -1
    for name, t in (("positions", positions), ("segments", segments)):
        _expect(name, t, (n,), torch.int32)
    for name, t, h in (("q", q, p.heads), ("k", k, p.kv_heads), ("v", v, p.kv_heads), ("out", out, p.heads)):
        _expect(name, t, (n, h, p.head_dim), _dt(p))
    w, nb = _ws(ws)
    _check(lib.pdattn_packed(ctypes.byref(p), n, _ptr(q), _ptr(k), _ptr(v), _ptr(positions), _ptr(segments),
                             _ptr(out), w, nb, _stream(stream)))


def packed_attend(p, v, positions, out, ws, stream=None):
    """Attention half of packed, over what its last call left in ws."""
    n = out.shape[0] if isinstance(out, torch.Tensor) else -1
    _expect("positions", positions, (n,), torch.int32)
    _expect("v", v, (n, p.kv_heads, p.head_dim), _dt(p))
    _expect("out", out, (n, p.heads, p.head_dim), _dt(p))
    w, nb = _ws(ws)
    _check(lib.pdattn_packed_attend(ctypes.byref(p), n, _ptr(v), _ptr(positions), _ptr(out), w, nb, _stream(stream)))


def check_status(ws, stream=None):
    """Synchronise, read and clear the device status; raise on a recorded error."""
    _check(lib.pdattn_check_status(_ptr(ws), _stream(stream)))


def last_launch_count():
    return int(lib.pdattn_last_launch_count())
