"""Pins for the oracle's paged prefill (CPU only).

The entry is the llama-3.1-8b-instruct page's ``prefill_paged`` (positions,
rows, slots per packed token, and the page table).  The oracle writes every
token's k and v at its slot, then attends each token over its row's cache.
Checked here against a dense numpy attention with an explicit causal mask,
causality, chunked prefill and the decode special case.
"""
import numpy as np
import pytest

import oracle
from paged_gqa_decode_step_gb300 import workloads as wl


def f64(a, od):
    return oracle.bf16_bits_to_f32(a).astype(np.float64) if od == oracle.BF16 else a.astype(np.float64)


def prep(w, seed=None):
    t = wl.generate_prefill(w, "cpu", seed=seed)
    a = {k: wl.to_numpy(v) for k, v in t.items()}
    od = oracle.BF16 if w.dtype == "bf16" else oracle.F32
    shape = oracle.make_shape(w.rows, w.heads, w.kv_heads, w.head_dim, w.pages_per_row, a["k_pool"].shape[0], od,
                              window=w.window, rope_theta=w.rope_theta)
    return a, shape, od


def run(a, shape, sinks=None):
    kp, vp = a["k_pool"].copy(), a["v_pool"].copy()
    q_rot, out, out64, rc = oracle.prefill_paged(shape, a["q"], a["k_new"], a["v_new"], a["positions"], a["rows"],
                                                 a["slots"], a["table"], kp, vp, sinks)
    assert rc == 0
    return q_rot, out, out64, kp, vp


W = wl.PrefillWorkload("p", prefix=(0, 70, 5), chunk=(40, 30, 64), heads=8, kv_heads=2, head_dim=64,
                       pages_per_row=3, dtype="f32", seed=3)


@pytest.mark.parametrize("window", [0, 50])
def test_prefill_matches_dense_causal_attention(window):
    w = wl.PrefillWorkload(**{**W.__dict__, "window": window})
    a, shape, od = prep(w)
    q_rot, _, out64, kp, vp = run(a, shape)
    g = w.heads // w.kv_heads
    for i in range(w.tokens):
        r, pos = int(a["rows"][i]), int(a["positions"][i])
        lo = max(0, pos - window + 1) if window > 0 else 0
        t = np.arange(lo, pos + 1)
        pages = a["table"][r, t // 64]
        K = f64(kp[pages, :, t % 64, :], od)          # [n, Hk, D]
        V = f64(vp[pages, :, t % 64, :], od)
        for h in range(w.heads):
            s = K[:, h // g] @ f64(q_rot[i, h], od) * 0.125
            pr = np.exp(s - s.max())
            pr /= pr.sum()
            assert np.abs(out64[i, h] - pr @ V[:, h // g]).max() <= 1e-12


def test_prefill_writes_every_token_at_its_slot():
    a, shape, od = prep(W)
    q_rot, _, _, kp, vp = run(a, shape)
    page, off = a["slots"] // 64, a["slots"] % 64
    assert np.array_equal(vp[page, :, off, :], a["v_new"])
    # the written k is the rotated k_new: the same rotation the queries get
    shape1 = oracle.make_shape(W.rows, W.kv_heads, W.kv_heads, W.head_dim, W.pages_per_row,
                               a["k_pool"].shape[0], od, rope_theta=W.rope_theta)
    kp2, vp2 = a["k_pool"].copy(), a["v_pool"].copy()
    k_rot, _, _, _ = oracle.prefill_paged(shape1, a["k_new"], a["k_new"], a["v_new"], a["positions"], a["rows"],
                                          a["slots"], a["table"], kp2, vp2)
    assert np.array_equal(kp[page, :, off, :], k_rot)


def test_later_tokens_never_reach_earlier_outputs():
    a, shape, od = prep(W)
    _, _, base, _, _ = run(a, shape)
    b = {k: v.copy() for k, v in a.items()}
    last = W.prefix[0] + W.chunk[0] - 1                 # last token of row 0
    i_last = int(np.where((a["rows"] == 0) & (a["positions"] == last))[0][0])
    b["k_new"][i_last] += np.float32(3.0)
    b["v_new"][i_last] -= np.float32(2.0)
    _, _, changed, _, _ = run(b, shape)
    row0 = np.where(a["rows"] == 0)[0]
    assert np.array_equal(base[row0[:-1]], changed[row0[:-1]])
    assert not np.array_equal(base[i_last], changed[i_last])


def test_chunked_prefill_equals_one_call():
    a, shape, od = prep(W)
    _, _, whole, kw, vw = run(a, shape)
    first = a["positions"] < np.array([W.prefix[r] for r in a["rows"]]) + 17
    kp, vp = a["k_pool"].copy(), a["v_pool"].copy()
    outs = np.zeros_like(whole)
    for sel in (first, ~first):
        idx = np.where(sel)[0]
        sub = {k: np.ascontiguousarray(a[k][idx]) for k in ("q", "k_new", "v_new", "positions", "rows", "slots")}
        _, _, o64, rc = oracle.prefill_paged(shape, sub["q"], sub["k_new"], sub["v_new"], sub["positions"],
                                             sub["rows"], sub["slots"], a["table"], kp, vp)
        assert rc == 0
        outs[idx] = o64
    assert np.array_equal(outs, whole)
    assert np.array_equal(kp, kw) and np.array_equal(vp, vw)


def test_one_token_per_row_is_decode():
    w = wl.PrefillWorkload("p1", prefix=(63, 100, 0), chunk=(1, 1, 1), heads=8, kv_heads=2, head_dim=64,
                           pages_per_row=3, dtype="bf16", seed=4)
    a, shape, od = prep(w)
    _, _, pre64, _, _ = run(a, shape)
    kp, vp = a["k_pool"].copy(), a["v_pool"].copy()
    _, _, dec64, rc = oracle.step(shape, a["q"], a["k_new"], a["v_new"], a["positions"], a["table"], kp, vp)
    assert rc == 0
    assert np.array_equal(pre64, dec64)
