"""Helpers for the GPU parity tests: run the CUDA path through the C-ABI and
the oracle on the same seeded inputs, and compare."""
import numpy as np
import torch

import oracle
from paged_gqa_decode_step_gb300 import workloads as wl

TOL = {"bf16": (2e-2, 2e-3), "f32": (1e-5, 1e-6)}   # (max |err|, mean |err|) vs the fp64 oracle


def binding():
    from paged_gqa_decode_step_gb300 import build
    build.build()
    from paged_gqa_decode_step_gb300 import binding as b
    return b


def oracle_shape(w, num_pages, rows=None):
    return oracle.make_shape(rows if rows is not None else w.rows, w.heads, w.kv_heads, w.head_dim,
                             w.pages_per_row, num_pages, oracle.BF16 if w.dtype == "bf16" else oracle.F32,
                             window=w.window, rope_theta=w.rope_theta)


def gpu_params(b, w, num_pages, tables, chunk_pages=0, rows=None, sinks=None):
    cos, sin = tables if tables is not None else (None, None)
    return b.make_params(rows if rows is not None else w.rows, w.heads, w.kv_heads, w.head_dim,
                         w.pages_per_row, num_pages, w.torch_dtype, window=w.window, rope_cos=cos,
                         rope_sin=sin, chunk_pages=chunk_pages, sinks=sinks)


def rope_tables_for(b, w):
    if w.rope_theta <= 0:
        return None
    return b.rope_tables(w.rope_theta, w.head_dim, w.max_seq, w.torch_dtype)


def as_f64(x, dtype):
    if dtype == "bf16":
        return oracle.bf16_bits_to_f32(x).astype(np.float64)
    return x.astype(np.float64)


def assert_close(got_t, want64, dtype, what=""):
    got = as_f64(wl.to_numpy(got_t), dtype)
    err = np.abs(got - want64)
    mx, mean = TOL[dtype]
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert err.max() <= mx, f"{what}: max |err| {err.max():.3g} > {mx}"
    assert err.mean() <= mean, f"{what}: mean |err| {err.mean():.3g} > {mean}"
    return err.max(), err.mean()


def run_step(w, poison=False, chunk_pages=0, mode="fused", seed=None, sinks=None):
    """One step on the GPU and in the oracle; returns the comparison data.
    sinks: None, or a list of per-head sink logits (rounded to the element type)."""
    b = binding()
    t = wl.generate(w, "cpu", poison=poison, seed=seed)
    a = {k: wl.to_numpy(v) for k, v in t.items()}
    num_pages = a["k_pool"].shape[0]
    kp, vp = a["k_pool"].copy(), a["v_pool"].copy()
    shape = oracle_shape(w, num_pages)
    sink_t = None
    if sinks is None:
        q_rot, _, out64, rc = oracle.step(shape, a["q"], a["k_new"], a["v_new"], a["positions"], a["table"], kp, vp)
        assert rc == 0
    else:
        sink_t = torch.tensor(sinks, dtype=torch.float32).to(w.torch_dtype)
        q_rot, rc = oracle.rope_write_kv(shape, a["q"], a["k_new"], a["v_new"], a["positions"], a["table"], kp, vp)
        assert rc == 0
        _, out64, rc = oracle.decode(shape, q_rot, a["positions"], a["table"], kp, vp, wl.to_numpy(sink_t))
        assert rc == 0
    d = {k: v.cuda() for k, v in t.items()}
    tables = rope_tables_for(b, w)
    p = gpu_params(b, w, num_pages, tables, chunk_pages, sinks=None if sink_t is None else sink_t.cuda())
    ws = b.new_workspace(p)
    out = torch.empty_like(d["q"])
    if mode == "fused":
        b.decode_fused(p, d["q"], d["k_new"], d["v_new"], d["positions"], d["table"], d["k_pool"],
                       d["v_pool"], out, ws)
    else:
        q_out = torch.empty_like(d["q"])
        b.rope_write_kv(p, d["q"], d["k_new"], d["v_new"], d["positions"], d["table"], q_out,
                        d["k_pool"], d["v_pool"], ws)
        b.decode(p, q_out, d["positions"], d["table"], d["k_pool"], d["v_pool"], out, ws)
        assert np.array_equal(wl.to_numpy(q_out).view(np.uint8), q_rot.view(np.uint8))
    b.check_status(ws)
    assert np.array_equal(wl.to_numpy(d["k_pool"]).view(np.uint8), kp.view(np.uint8)), "k pool differs"
    assert np.array_equal(wl.to_numpy(d["v_pool"]).view(np.uint8), vp.view(np.uint8)), "v pool differs"
    return assert_close(out, out64, w.dtype, w.name)
