"""Pins for the oracle's packed attention (CPU only).

Llama example page, "src/attention.linnet", `packed`: sequences packed into
one row, each token rotated at its own position and attending to the tokens
of its own sequence at positions up to its own.  Checked against textbook
causal attention (one sequence), segment isolation, invariance under the
order of the packed tokens, the oracle's paged prefill on an empty cache, a
banded window, and a closed form for sinks.
"""
import numpy as np
import pytest

import oracle
from paged_gqa_decode_step_gb300 import workloads as wl


def f64(a, od):
    return oracle.bf16_bits_to_f32(a).astype(np.float64) if od == oracle.BF16 else a.astype(np.float64)


def prep(w):
    t = wl.generate_packed(w, "cpu")
    a = {k: wl.to_numpy(v) for k, v in t.items()}
    od = oracle.BF16 if w.dtype == "bf16" else oracle.F32
    shape = oracle.make_shape(0, w.heads, w.kv_heads, w.head_dim, 1, 1, od, window=w.window, rope_theta=w.rope_theta)
    return a, shape, od


def run(a, shape, sinks=None):
    q_rot, k_rot, out, out64, rc = oracle.packed(shape, a["q"], a["k"], a["v"], a["positions"], a["segments"], sinks)
    assert rc == 0
    return q_rot, k_rot, out, out64


def dense_causal(q_rot, k_rot, v, g, band=0):
    """Textbook causal softmax attention over one contiguous sequence (numpy)."""
    n, Hq, D = q_rot.shape
    kk = np.repeat(k_rot, g, axis=1)
    vv = np.repeat(v, g, axis=1)
    s = np.einsum("ihd,jhd->hij", q_rot, kk) * np.float32(1 / np.sqrt(D)).astype(np.float64)
    i, j = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
    mask = j <= i
    if band:
        mask &= j > i - band
    s = np.where(mask[None], s, -np.inf)
    p = np.exp(s - s.max(axis=2, keepdims=True))
    p /= p.sum(axis=2, keepdims=True)
    return np.einsum("hij,jhd->ihd", p, vv)


@pytest.mark.parametrize("dtype,window", [("f32", 0), ("bf16", 0), ("f32", 20)])
def test_one_sequence_is_causal_attention(dtype, window):
    w = wl.PackedWorkload("one", lengths=(70,), heads=8, kv_heads=2, head_dim=64, dtype=dtype, window=window, seed=1)
    a, shape, od = prep(w)
    q_rot, k_rot, _, out64 = run(a, shape)
    want = dense_causal(f64(q_rot, od), f64(k_rot, od), f64(a["v"], od), 4, band=window)
    assert np.abs(out64 - want).max() <= 1e-12


def test_sequences_do_not_see_each_other():
    w = wl.PackedWorkload("two", lengths=(40, 25, 33), heads=4, kv_heads=2, head_dim=64, dtype="f32", seed=2)
    a, shape, od = prep(w)
    _, _, _, whole = run(a, shape)
    start = 0
    for L in w.lengths:
        sub = {k: np.ascontiguousarray(v[start:start + L]) for k, v in a.items()}
        _, _, _, alone = run(sub, shape)
        assert np.array_equal(alone, whole[start:start + L])
        start += L


def test_token_order_in_the_pack_does_not_matter():
    w = wl.PackedWorkload("order", lengths=(30, 20, 14), heads=8, kv_heads=4, head_dim=64, dtype="bf16",
                          shuffle_ids=True, seed=3)
    a, shape, od = prep(w)
    _, _, _, base = run(a, shape)
    perm = np.random.default_rng(3).permutation(w.tokens)
    b = {k: np.ascontiguousarray(v[perm]) for k, v in a.items()}
    _, _, _, shuffled = run(b, shape)
    assert np.abs(shuffled - base[perm]).max() <= 1e-13


def test_packed_sequence_equals_prefill_of_an_empty_row():
    # the same tokens as a prefill into row 0 of a cache (pages 0 .. 2 in order)
    w = wl.PackedWorkload("pf", lengths=(150,), heads=8, kv_heads=2, head_dim=64, dtype="bf16", seed=4)
    a, shape, od = prep(w)
    _, _, _, out64 = run(a, shape)
    n = w.tokens
    pshape = oracle.make_shape(1, w.heads, w.kv_heads, w.head_dim, 3, 3, od, rope_theta=w.rope_theta)
    zeros = np.zeros((3, w.kv_heads, 64, w.head_dim), np.uint16)
    rows = np.zeros(n, np.int32)
    slots = np.arange(n, dtype=np.int32)
    table = np.arange(3, dtype=np.int32)[None]
    _, _, pf64, rc = oracle.prefill_paged(pshape, a["q"], a["k"], a["v"], a["positions"], rows, slots, table,
                                          zeros.copy(), zeros.copy())
    assert rc == 0
    assert np.abs(pf64 - out64).max() <= 1e-12


def test_sinks_scale_by_the_closed_form():
    # with a sink s: out = out_without * Z / (Z + e^s), Z = sum over visible keys of e^score
    w = wl.PackedWorkload("sinks", lengths=(20, 9), heads=4, kv_heads=2, head_dim=64, dtype="f32", seed=5)
    a, shape, od = prep(w)
    q_rot, k_rot, _, base = run(a, shape)
    sinks = np.array([0.5, -1.0, 2.0, 0.0], np.float32)
    _, _, _, with_sink = run(a, shape, sinks)
    scale = float(np.float32(1 / np.sqrt(64)))
    for i in range(w.tokens):
        for h in range(4):
            js = [j for j in range(w.tokens) if a["segments"][j] == a["segments"][i] and
                  a["positions"][j] <= a["positions"][i]]
            z = sum(np.exp(scale * np.dot(q_rot[i, h].astype(np.float64), k_rot[j, h // 2].astype(np.float64)))
                    for j in js)
            assert np.allclose(with_sink[i, h], base[i, h] * z / (z + np.exp(float(sinks[h]))), rtol=1e-12,
                               atol=1e-14)
