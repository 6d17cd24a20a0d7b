"""Pins for the oracle's cache write and attention (CPU only).

The oracle follows the Llama example page, ``src/attention.linnet``
(``decode``): write k and v at pos, mask ``seen[s] = s <= pos``, scale
``rsqrt(f32(H / Heads))``, grouped attention where query head h reads kv head
h / (Heads / KvHeads) ("Key ideas", grouped-query attention); the page slot
comes from the ``decode_paged`` signature on the llama-3.1-8b-instruct page
(``table: Tensor[Rows, Pages; i32]``, ``PageSize = 64``) and the window from
the gpt-oss-20b page (``window: i32``).  Every test here checks the oracle
against something other than its own code: a dense numpy / torch attention
over a cache rebuilt contiguously through the table, closed forms, exact
special cases and invariances.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_step_gb300 import workloads as wl


def f64(a, dtype):
    return oracle.bf16_bits_to_f32(a).astype(np.float64) if dtype == oracle.BF16 else a.astype(np.float64)


def case(R=3, Hq=8, Hk=2, D=64, Pg=6, dtype="bf16", positions=(0, 64, 300), window=0,
         theta=10000.0, seed=7, poison=False, num_pages=0):
    w = wl.Workload("t", rows=R, heads=Hq, kv_heads=Hk, head_dim=D, pages_per_row=Pg, dtype=dtype,
                    rope_theta=theta, window=window, positions="fixed", fixed_positions=tuple(positions),
                    num_pages=num_pages, seed=seed)
    t = wl.generate(w, "cpu", poison=poison)
    a = {k: wl.to_numpy(v) for k, v in t.items()}
    od = oracle.BF16 if dtype == "bf16" else oracle.F32
    shape = oracle.make_shape(R, Hq, Hk, D, Pg, a["k_pool"].shape[0], od, window=window, rope_theta=theta)
    return w, a, shape, od


def contiguous_cache(a, shape):
    """[R, Hk, Pg*64, D] cache gathered through the table with numpy indexing."""
    table = a["table"]
    R, Pg = table.shape
    t = np.arange(Pg * 64)
    pages = table[:, t // 64]                      # [R, S]
    safe = np.where(pages >= 0, pages, 0)
    K = a["k_pool"][safe, :, (t % 64)[None, :], :]  # [R, S, Hk, D]
    V = a["v_pool"][safe, :, (t % 64)[None, :], :]
    return np.ascontiguousarray(K.transpose(0, 2, 1, 3)), np.ascontiguousarray(V.transpose(0, 2, 1, 3))


def dense_attention(q, K, V, positions, window, scale, group):
    """softmax(q K^T * scale + mask) V in float64 with numpy einsum."""
    R, Hq, D = q.shape
    S = K.shape[2]
    out = np.zeros((R, Hq, D))
    t = np.arange(S)
    for r in range(R):
        pos = positions[r]
        lo = max(0, pos - window + 1) if window > 0 else 0
        mask = (t <= pos) & (t >= lo)
        Kr = np.repeat(K[r], group, axis=0)         # [Hq, S, D]
        Vr = np.repeat(V[r], group, axis=0)
        s = np.einsum("hd,hsd->hs", q[r], Kr) * scale
        s = np.where(mask[None, :], s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        out[r] = np.einsum("hs,hsd->hd", np.where(mask[None, :], p, 0.0), np.where(mask[None, :, None], Vr, 0.0))
    return out


SCALE = {64: 0.125, 128: float(np.float32(1.0 / math.sqrt(128.0)))}


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("Hq,Hk,D,window", [(8, 2, 64, 0), (8, 8, 64, 0), (16, 2, 128, 0),
                                             (8, 1, 64, 100), (4, 4, 128, 64)])
def test_decode_matches_dense_attention(dtype, Hq, Hk, D, window):
    w, a, shape, od = case(Hq=Hq, Hk=Hk, D=D, dtype=dtype, window=window, positions=(0, 64, 300))
    q_rot, _ = oracle.rope_write_kv(shape, a["q"], a["k_new"], a["v_new"], a["positions"],
                                    a["table"], a["k_pool"], a["v_pool"])
    out, out64, rc = oracle.decode(shape, q_rot, a["positions"], a["table"], a["k_pool"], a["v_pool"])
    assert rc == 0
    K, V = contiguous_cache(a, shape)
    want = dense_attention(f64(q_rot, od), f64(K, od), f64(V, od), a["positions"], window,
                           SCALE[D], Hq // Hk)
    assert np.abs(out64 - want).max() <= 1e-12


def test_decode_matches_torch_sdpa_gqa():
    # A second library route: torch's scaled_dot_product_attention in float64
    # with repeat_interleave for the groups and an explicit boolean mask.
    w, a, shape, od = case(R=2, Hq=32, Hk=8, D=128, Pg=4, positions=(130, 255), theta=500000.0)
    out, out64, rc = oracle.decode(shape, a["q"], a["positions"], a["table"], a["k_pool"], a["v_pool"])
    assert rc == 0
    K, V = contiguous_cache(a, shape)
    for r in range(2):
        pos = int(a["positions"][r])
        q = torch.from_numpy(f64(a["q"][r], od))[:, None, :]           # [Hq, 1, D]
        k = torch.from_numpy(f64(K[r, :, : pos + 1], od)).repeat_interleave(4, dim=0)
        v = torch.from_numpy(f64(V[r, :, : pos + 1], od)).repeat_interleave(4, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=SCALE[128])[:, 0, :]
        assert np.abs(out64[r] - ref.numpy()).max() <= 1e-12


def test_page_placement_does_not_matter():
    # Identity table vs shuffled table over the same logical cache: identical.
    w, a, shape, od = case(R=2, Hq=8, Hk=2, D=64, Pg=5, positions=(200, 319))
    out_a, o64_a, _ = oracle.decode(shape, a["q"], a["positions"], a["table"], a["k_pool"], a["v_pool"])
    K, V = contiguous_cache(a, shape)     # [R, Hk, S, D]
    R, Hk, S, D = K.shape
    ident_k = np.ascontiguousarray(K.reshape(R, Hk, S // 64, 64, D).transpose(0, 2, 1, 3, 4).reshape(-1, Hk, 64, D))
    ident_v = np.ascontiguousarray(V.reshape(R, Hk, S // 64, 64, D).transpose(0, 2, 1, 3, 4).reshape(-1, Hk, 64, D))
    ident_t = np.arange(R * (S // 64), dtype=np.int32).reshape(R, S // 64)
    shape2 = oracle.make_shape(R, 8, 2, 64, S // 64, ident_k.shape[0], od)
    out_b, o64_b, rc = oracle.decode(shape2, a["q"], a["positions"], ident_t, ident_k, ident_v)
    assert rc == 0
    assert np.array_equal(o64_a, o64_b) and np.array_equal(out_a, out_b)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_single_visible_position_returns_v(dtype):
    # pos = 0 (and any pos with window 1): the only weight is exactly 1.
    w, a, shape, od = case(R=2, Hq=8, Hk=2, dtype=dtype, positions=(0, 150))
    shape.window = 1
    q_rot, _ = oracle.rope_write_kv(shape, a["q"], a["k_new"], a["v_new"], a["positions"],
                                    a["table"], a["k_pool"], a["v_pool"])
    out, out64, rc = oracle.decode(shape, q_rot, a["positions"], a["table"], a["k_pool"], a["v_pool"])
    assert rc == 0
    want = np.repeat(a["v_new"], 4, axis=1)
    assert np.array_equal(out, want)


def test_constant_values_give_that_constant():
    w, a, shape, od = case(R=2, Hq=8, Hk=2, D=64, positions=(77, 299))
    const = np.linspace(-2, 2, 64).astype(np.float32)
    bits = torch.from_numpy(const).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    a["v_pool"][:] = bits
    out, out64, rc = oracle.decode(shape, a["q"], a["positions"], a["table"], a["k_pool"], a["v_pool"])
    assert rc == 0
    assert np.abs(out64 - f64(bits, od)[None, None, :]).max() <= 1e-12
    assert np.all(out == bits[None, None, :])


def test_weights_are_the_closed_form_softmax_and_sum_to_one():
    # V[t] = one-hot(t) turns the output into the weight vector; with q = a*e0
    # and K[t] = b_t*e0 the scores are scale*a*b_t, so the weights are the
    # closed-form softmax of those.
    R, Hq, Hk, D, pos = 1, 4, 1, 64, 40
    shape = oracle.make_shape(R, Hq, Hk, D, 1, 1, oracle.F32)
    q = np.zeros((R, Hq, D), np.float32)
    q[0, :, 0] = [0.5, 1.0, 2.0, -3.0]
    b = np.linspace(-1, 1, 64).astype(np.float32)
    kp = np.zeros((1, 1, 64, D), np.float32)
    kp[0, 0, :, 0] = b
    vp = np.zeros((1, 1, 64, D), np.float32)
    vp[0, 0, np.arange(64), np.arange(64)] = 1.0
    table = np.zeros((1, 1), np.int32)
    _, out64, rc = oracle.decode(shape, q, np.array([pos], np.int32), table, kp, vp)
    assert rc == 0
    for h in range(Hq):
        s = 0.125 * float(q[0, h, 0]) * b[: pos + 1].astype(np.float64)
        p = np.exp(s - s.max())
        p /= p.sum()
        assert np.abs(out64[0, h, : pos + 1] - p).max() <= 1e-15
        assert np.all(out64[0, h, pos + 1:] == 0.0)
        assert abs(out64[0, h].sum() - 1.0) <= 1e-12


def test_score_shift_invariance():
    # Adding alpha*e_j to every cached key adds alpha*q_j to every score of a
    # head: softmax is unchanged.
    w, a, shape, od = case(R=2, Hq=4, Hk=4, D=64, dtype="f32", positions=(33, 170))
    _, base, _ = oracle.decode(shape, a["q"], a["positions"], a["table"], a["k_pool"], a["v_pool"])
    kp = a["k_pool"].copy()
    kp[..., 5] += np.float32(0.75)
    _, shifted, _ = oracle.decode(shape, a["q"], a["positions"], a["table"], kp, a["v_pool"])
    # the f32 keys round when shifted, so compare at f32 input precision
    assert np.abs(base - shifted).max() <= 1e-4


def test_group_mapping_uses_h_div_group():
    # kv head j holds constant values j+1: query head h must return h//g + 1.
    R, Hq, Hk, D = 1, 8, 2, 64
    w, a, shape, od = case(R=1, Hq=Hq, Hk=Hk, D=D, dtype="f32", positions=(90,))
    for j in range(Hk):
        a["v_pool"][:, j] = np.float32(j + 1)
    _, out64, _ = oracle.decode(shape, a["q"], a["positions"], a["table"], a["k_pool"], a["v_pool"])
    for h in range(Hq):
        assert np.abs(out64[0, h] - (h // (Hq // Hk) + 1)).max() <= 1e-12


def test_window_at_least_context_equals_full():
    w, a, shape, od = case(positions=(10, 64, 300))
    _, full, _ = oracle.decode(shape, a["q"], a["positions"], a["table"], a["k_pool"], a["v_pool"])
    shape.window = 301
    _, win, _ = oracle.decode(shape, a["q"], a["positions"], a["table"], a["k_pool"], a["v_pool"])
    assert np.array_equal(full, win)
    shape.window = 300                         # row 2 now drops position 0
    _, win2, _ = oracle.decode(shape, a["q"], a["positions"], a["table"], a["k_pool"], a["v_pool"])
    assert np.array_equal(full[:2], win2[:2]) and not np.array_equal(full[2], win2[2])


def test_unreadable_slots_are_never_read():
    # Spare pages, slots past pos and slots before the window hold NaN.
    w, a, shape, od = case(R=3, Hq=8, Hk=2, positions=(5, 130, 383), window=70, poison=True, num_pages=12)
    q_rot, rc = oracle.rope_write_kv(shape, a["q"], a["k_new"], a["v_new"], a["positions"],
                                     a["table"], a["k_pool"], a["v_pool"])
    out, out64, rc2 = oracle.decode(shape, q_rot, a["positions"], a["table"], a["k_pool"], a["v_pool"])
    assert rc == 0 and rc2 == 0 and np.all(np.isfinite(out64))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_cache_write_is_the_paged_scatter(dtype):
    # Without rotation the written slot is k_new / v_new bit for bit; with
    # rotation it equals the rotated q of the same vector.  Nothing else in
    # the pools changes.  The expected pools come from numpy fancy indexing.
    w, a, shape, od = case(R=3, Hq=2, Hk=2, D=64, dtype=dtype, positions=(0, 63, 64 * 4 + 17), theta=0.0)
    kp0, vp0 = a["k_pool"].copy(), a["v_pool"].copy()
    _, rc = oracle.rope_write_kv(shape, a["q"], a["k_new"], a["v_new"], a["positions"], a["table"],
                                 a["k_pool"], a["v_pool"])
    assert rc == 0
    pos = a["positions"].astype(np.int64)
    pages = a["table"][np.arange(3), pos // 64]
    kp0[pages, :, pos % 64, :] = a["k_new"]
    vp0[pages, :, pos % 64, :] = a["v_new"]
    assert np.array_equal(kp0.view(np.uint8), a["k_pool"].view(np.uint8))
    assert np.array_equal(vp0.view(np.uint8), a["v_pool"].view(np.uint8))
    # rotated: same vectors through q and through k give the same bits
    w, a, shape, od = case(R=3, Hq=2, Hk=2, D=64, dtype=dtype, positions=(0, 63, 64 * 4 + 17), theta=10000.0)
    q_rot, _ = oracle.rope_write_kv(shape, a["k_new"], a["k_new"], a["v_new"], a["positions"],
                                    a["table"], a["k_pool"], a["v_pool"])
    pages = a["table"][np.arange(3), pos // 64]
    assert np.array_equal(a["k_pool"][pages, :, pos % 64, :].view(np.uint8), q_rot.view(np.uint8))


def test_errors_are_reported():
    w, a, shape, od = case(positions=(0, 64, 300))
    bad = a["positions"].copy()
    bad[1] = 6 * 64                      # past the table
    _, _, rc = oracle.decode(shape, a["q"], bad, a["table"], a["k_pool"], a["v_pool"])
    assert rc == 1
    tab = a["table"].copy()
    tab[2, 1] = 10 ** 6                  # page id outside the pool
    _, _, rc = oracle.decode(shape, a["q"], a["positions"], tab, a["k_pool"], a["v_pool"])
    assert rc == 4


def test_split_merge_of_any_partition_reproduces_the_whole():
    # The flash-decoding merge the GPU uses: for any partition of the visible
    # positions into chunks with (m_j, l_j, o_j) = (max, sum exp(s - m_j),
    # sum exp(s - m_j) v), out = sum_j e^{m_j - M} o_j / sum_j e^{m_j - M} l_j.
    w, a, shape, od = case(R=1, Hq=4, Hk=1, D=64, Pg=6, positions=(333,), dtype="f32")
    _, out64, _ = oracle.decode(shape, a["q"], a["positions"], a["table"], a["k_pool"], a["v_pool"])
    K, V = contiguous_cache(a, shape)
    q = a["q"][0].astype(np.float64)
    s = np.einsum("hd,sd->hs", q, K[0, 0, :334].astype(np.float64)) * 0.125
    rng = np.random.default_rng(1)
    for _ in range(5):
        cuts = np.sort(rng.choice(np.arange(1, 334), size=rng.integers(1, 8), replace=False))
        bounds = [0, *cuts.tolist(), 334]
        parts = []
        for lo, hi in zip(bounds[:-1], bounds[1:]):
            m = s[:, lo:hi].max(axis=1)
            e = np.exp(s[:, lo:hi] - m[:, None])
            parts.append((m, e.sum(axis=1), e @ V[0, 0, lo:hi].astype(np.float64)))
        M = np.max([p[0] for p in parts], axis=0)
        num = sum(np.exp(p[0] - M)[:, None] * p[2] for p in parts)
        den = sum(np.exp(p[0] - M) * p[1] for p in parts)
        assert np.abs(num / den[:, None] - out64[0]).max() <= 1e-12


# ---- attention sinks (gpt-oss-20b page, SinkAttention `param sinks`) ------
def test_sink_at_minus_infinity_changes_nothing():
    w, a, shape, od = case(R=2, Hq=8, Hk=2, D=64, dtype="f32", positions=(40, 300))
    _, base, _ = oracle.decode(shape, a["q"], a["positions"], a["table"], a["k_pool"], a["v_pool"])
    sinks = np.full(8, -np.inf, dtype=np.float32)
    _, with_sink, _ = oracle.decode(shape, a["q"], a["positions"], a["table"], a["k_pool"], a["v_pool"], sinks)
    assert np.array_equal(base, with_sink)


def test_sink_weights_closed_form():
    # With every score equal (q = 0) each of the n visible positions weighs
    # 1 / (n + e^(sink - 0)) and the sink takes the rest; V = one-hot rows
    # expose the weights.
    R, Hq, Hk, D, pos = 1, 4, 1, 64, 50
    shape = oracle.make_shape(R, Hq, Hk, D, 1, 1, oracle.F32)
    q = np.zeros((R, Hq, D), np.float32)
    kp = np.random.default_rng(0).standard_normal((1, 1, 64, D)).astype(np.float32)
    vp = np.zeros((1, 1, 64, D), np.float32)
    vp[0, 0, np.arange(64), np.arange(64)] = 1.0
    sinks = np.array([-2.0, 0.0, 1.5, 4.0], np.float32)
    _, out64, rc = oracle.decode(shape, q, np.array([pos], np.int32), np.zeros((1, 1), np.int32), kp, vp, sinks)
    assert rc == 0
    n = pos + 1
    for h in range(Hq):
        wgt = 1.0 / (n + math.exp(float(sinks[h])))
        assert np.abs(out64[0, h, :n] - wgt).max() <= 1e-15
        assert abs(out64[0, h].sum() - n * wgt) <= 1e-12


def test_sinks_against_dense_reference():
    w, a, shape, od = case(R=3, Hq=16, Hk=4, D=64, dtype="bf16", positions=(0, 70, 380), window=100)
    rng = np.random.default_rng(4)
    sinks = torch.from_numpy(rng.standard_normal(16).astype(np.float32)).to(torch.bfloat16)
    sb = sinks.view(torch.int16).numpy().view(np.uint16)
    _, out64, rc = oracle.decode(shape, a["q"], a["positions"], a["table"], a["k_pool"], a["v_pool"], sb)
    assert rc == 0
    K, V = contiguous_cache(a, shape)
    q = f64(a["q"], od)
    Kf, Vf = f64(K, od), f64(V, od)
    S = Kf.shape[2]
    t = np.arange(S)
    for r in range(3):
        pos = int(a["positions"][r])
        lo = max(0, pos - 100 + 1)
        mask = (t <= pos) & (t >= lo)
        for h in range(16):
            s = (Kf[r, h // 4] @ q[r, h]) * 0.125
            logits = np.concatenate([s[mask], [float(sinks[h])]])
            p = np.exp(logits - logits.max())
            p /= p.sum()
            want = p[:-1] @ Vf[r, h // 4][mask]
            assert np.abs(out64[r, h] - want).max() <= 1e-12
