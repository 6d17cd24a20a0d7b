"""Pins for the oracle's rotary tables and RoPE (CPU only).

The tables follow the Llama example page, ``src/rope.linnet`` (``tables``):
inv_freq[i] = exp(-(2i / D) * ln theta), angle = s * inv_freq, the halves of
the head dimension repeat the same frequencies, cos and sin cast to T.  These
tests check the oracle against what that definition fixes independently of
its code: exact special cases, high-precision closed forms within a derived
error bound, a dense rotation matrix, and the rotation invariants.
"""
import math

import mpmath
import numpy as np
import pytest
import torch

import oracle

mpmath.mp.dps = 40


def bf16_of(x64: np.ndarray) -> np.ndarray:
    """float64 -> f32 -> bf16 bits via torch's round-to-nearest-even."""
    t = torch.from_numpy(np.asarray(x64, dtype=np.float64)).to(torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def f32(bits):
    return oracle.bf16_bits_to_f32(bits).astype(np.float64)


@pytest.mark.parametrize("theta,D", [(10000.0, 64), (500000.0, 128), (150000.0, 64)])
def test_position_zero_is_identity_rotation(theta, D):
    c, s = oracle.rope_tables(theta, D, 4, oracle.BF16)
    assert np.all(c[0] == 0x3F80)          # bf16 1.0
    assert np.all(s[0] == 0)               # +0.0
    c32, s32 = oracle.rope_tables(theta, D, 4, oracle.F32)
    assert np.all(c32[0] == 1.0) and np.all(s32[0] == 0.0)


@pytest.mark.parametrize("theta,D", [(10000.0, 64), (500000.0, 128)])
def test_halves_share_frequencies(theta, D):
    # full = concat(angles, angles): column i and i + D/2 are equal.
    c, s = oracle.rope_tables(theta, D, 300, oracle.BF16)
    assert np.array_equal(c[:, : D // 2], c[:, D // 2:])
    assert np.array_equal(s[:, : D // 2], s[:, D // 2:])


def test_first_frequency_is_plain_cos_of_position():
    # inv_freq[0] = exp(-0 * ln theta) = 1 exactly, so angle = s exactly and
    # column 0 is cos(s), sin(s) rounded f32 -> bf16.  Checked bit for bit
    # against 40-digit mpmath values.
    S = 8192
    c, s = oracle.rope_tables(500000.0, 128, S, oracle.BF16)
    want_c = bf16_of(np.array([float(mpmath.cos(k)) for k in range(S)]))
    want_s = bf16_of(np.array([float(mpmath.sin(k)) for k in range(S)]))
    assert np.array_equal(c[:, 0], want_c)
    assert np.array_equal(s[:, 0], want_s)
    c32, s32 = oracle.rope_tables(500000.0, 128, S, oracle.F32)
    assert np.array_equal(c32[:, 0], np.array([float(mpmath.cos(k)) for k in range(S)], dtype=np.float32))


@pytest.mark.parametrize("theta,D,S", [(10000.0, 64, 512), (500000.0, 128, 8192), (150000.0, 64, 4096)])
def test_every_frequency_within_closed_form_bound(theta, D, S):
    # Exact value: cos(s * theta**(-2i/D)).  The f32 pipeline of the pages
    # (2i/D, ln theta, their product, exp, times s) perturbs the angle by at
    # most s * inv_freq * (|arg| + 3) * 2^-24 + ulp(angle); cos/sin move by at
    # most that much, and the bf16 cast adds half a bf16 ulp (2^-9 relative,
    # at most 2^-9 absolute for |x| <= 1).
    c, s = oracle.rope_tables(theta, D, S, oracle.F32)
    half = D // 2
    pos = np.arange(S, dtype=np.float64)[:, None]
    i = np.arange(half, dtype=np.float64)[None, :]
    inv = np.array([float(mpmath.power(theta, -mpmath.mpf(2 * k) / D)) for k in range(half)])[None, :]
    ang = pos * inv
    arg = 2 * i / D * math.log(theta)
    bound = ang * (arg + 3.0) * 2.0 ** -24 + np.abs(ang) * 2.0 ** -24 + 2.0 ** -24
    assert np.all(np.abs(c[:, :half] - np.cos(ang)) <= bound + 1e-12)
    assert np.all(np.abs(s[:, :half] - np.sin(ang)) <= bound + 1e-12)
    cb, sb = oracle.rope_tables(theta, D, S, oracle.BF16)
    assert np.all(np.abs(f32(cb[:, :half]) - np.cos(ang)) <= bound + 2.0 ** -9)
    assert np.all(np.abs(f32(sb[:, :half]) - np.sin(ang)) <= bound + 2.0 ** -9)


def test_pythagorean_identity():
    c, s = oracle.rope_tables(500000.0, 128, 2048, oracle.BF16)
    r = f32(c) ** 2 + f32(s) ** 2
    assert np.all(np.abs(r - 1.0) <= 2 * 2.0 ** -8)


def _rope_f32(x, pos, theta):
    """Run the oracle's rope on vectors x [n, D] (f32) at one position."""
    n, D = x.shape
    shape = oracle.make_shape(rows=1, heads=n, kv_heads=n, head_dim=D, pages_per_row=pos // 64 + 1,
                              num_pages=pos // 64 + 1, dtype=oracle.F32, rope_theta=theta)
    q = np.ascontiguousarray(x[None].astype(np.float32))
    kp = np.zeros((pos // 64 + 1, n, 64, D), np.float32)
    vp = np.zeros_like(kp)
    table = np.arange(pos // 64 + 1, dtype=np.int32)[None]
    q_out, rc = oracle.rope_write_kv(shape, q, q[0].copy()[None], q[0].copy()[None],
                                     np.array([pos], np.int32), table, kp, vp)
    assert rc == 0
    return q_out[0].astype(np.float64), kp[table[0, pos // 64], :, pos % 64, :].astype(np.float64)


def _rotation_matrix(D, pos, theta):
    half = D // 2
    M = np.zeros((D, D))
    for i in range(half):
        a = float(mpmath.mpf(pos) * mpmath.power(theta, -mpmath.mpf(2 * i) / D))
        c, s = math.cos(a), math.sin(a)
        M[i, i] = c
        M[i, i + half] = -s
        M[i + half, i] = s
        M[i + half, i + half] = c
    return M


@pytest.mark.parametrize("D,theta", [(64, 10000.0), (128, 500000.0)])
@pytest.mark.parametrize("pos", [1, 7, 63, 100])
def test_rope_is_the_dense_rotation(D, theta, pos):
    # y = M x with M the block rotation pairing dim i with i + D/2 (the
    # rotate_half convention); the written k slot gets the same rotation.
    rng = np.random.default_rng(pos * 7 + D)
    x = rng.standard_normal((3, D)).astype(np.float32)
    y, kslot = _rope_f32(x, pos, theta)
    want = x.astype(np.float64) @ _rotation_matrix(D, pos, theta).T
    tol = 1e-5 * (1 + pos) * np.abs(x).max()
    assert np.abs(y - want).max() <= tol
    assert np.array_equal(kslot.astype(np.float32), y.astype(np.float32))


def test_rope_preserves_pair_norms():
    D = 128
    rng = np.random.default_rng(5)
    x = rng.standard_normal((4, D)).astype(np.float32)
    y, _ = _rope_f32(x, 777, 500000.0)
    h = D // 2
    nx = x[:, :h].astype(np.float64) ** 2 + x[:, h:].astype(np.float64) ** 2
    ny = y[:, :h] ** 2 + y[:, h:] ** 2
    assert np.abs(nx - ny).max() <= 1e-5 * nx.max()


def test_rope_scores_depend_on_relative_position_only():
    # <R_m q, R_n k> = <R_{m+d} q, R_{n+d} k>: the property RoPE exists for.
    D = 64
    rng = np.random.default_rng(11)
    q = rng.standard_normal((1, D)).astype(np.float32)
    k = rng.standard_normal((1, D)).astype(np.float32)
    base = None
    for shift in (0, 5, 40, 90):
        qm, _ = _rope_f32(q, 10 + shift, 10000.0)
        kn, _ = _rope_f32(k, 3 + shift, 10000.0)
        dot = float(qm[0] @ kn[0])
        if base is None:
            base = dot
        assert abs(dot - base) <= 1e-4 * (1 + abs(base))


def test_bf16_rope_is_rotation_within_rounding():
    # bf16 inputs, bf16 tables, one rounding of the result: within a few bf16
    # ulps of the exact rotation of the same inputs.
    D, pos, theta = 128, 3000, 500000.0
    rng = np.random.default_rng(3)
    x32 = rng.standard_normal((8, D)).astype(np.float32)
    xb = bf16_of(x32)
    shape = oracle.make_shape(rows=1, heads=8, kv_heads=8, head_dim=D, pages_per_row=pos // 64 + 1,
                              num_pages=pos // 64 + 1, dtype=oracle.BF16, rope_theta=theta)
    kp = np.zeros((pos // 64 + 1, 8, 64, D), np.uint16)
    table = np.arange(pos // 64 + 1, dtype=np.int32)[None]
    q_out, rc = oracle.rope_write_kv(shape, xb[None].copy(), xb[None].copy(), xb[None].copy(),
                                     np.array([pos], np.int32), table, kp, kp.copy())
    assert rc == 0
    y = f32(q_out[0])
    x = f32(xb)
    want = x @ _rotation_matrix(D, pos, theta).T
    # y_j = x_j c_j -/+ x_pair s_j: each table entry is within 2^-9 (bf16
    # cast) plus the angle perturbation of the f32 pipeline of its exact
    # value, and the result is rounded once more to bf16.
    h = D // 2
    i = np.arange(h)
    ang = pos * theta ** (-2.0 * i / D)
    d_ang = ang * (2 * i / D * math.log(theta) + 4.0) * 2.0 ** -24 + 2.0 ** -24
    e_tab = np.concatenate([d_ang, d_ang]) + 2.0 ** -9
    pair = np.concatenate([x[:, h:], x[:, :h]], axis=1)
    bound = (np.abs(x) + np.abs(pair)) * e_tab + np.abs(want) * 2.0 ** -8 + 1e-6
    assert np.all(np.abs(y - want) <= bound)


def test_bf16_rounding_helper_ties_to_even():
    # 1 + 2^-8 is exactly between bf16 1.0 and 1 + 2^-7: ties to the even 1.0;
    # 1 + 3*2^-8 ties to 1 + 2^-6 (even mantissa).
    assert oracle.f32_to_bf16_bits(1.0 + 2.0 ** -8) == 0x3F80
    assert oracle.f32_to_bf16_bits(1.0 + 3 * 2.0 ** -8) == 0x3F82
    assert oracle.f32_to_bf16_bits(-2.5) == 0xC020
    x = np.random.default_rng(0).standard_normal(10000).astype(np.float32)
    want = bf16_of(x.astype(np.float64))
    got = np.array([oracle.f32_to_bf16_bits(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, want)


def test_bf16_rope_uses_tables_cast_to_T():
    # The tables are cast to T before rope uses them (`cast<T>(cos(full))`).
    # For x = a*e_0 the rotation gives y_0 = bf16(a * C), y_{D/2} = bf16(a * S)
    # with C, S the bf16 roundings of cos(pos), sin(pos) (column 0 has
    # inv_freq = 1).  Products of two bf16 values are exact in float64; the
    # expected bits come from 40-digit mpmath and torch's rounding only.
    D, theta = 64, 10000.0
    positions = np.arange(0, 4096, 7)
    scales = np.array([1.5, -1.171875, 3.3125, 0.80078125], dtype=np.float32)   # bf16-exact
    R, Hq = len(positions), len(scales)
    q = np.zeros((R, Hq, D), np.float32)
    q[:, :, 0] = scales[None, :]
    qb = bf16_of(q)
    Pg = 4096 // 64
    shape = oracle.make_shape(rows=R, heads=Hq, kv_heads=1, head_dim=D, pages_per_row=Pg,
                              num_pages=Pg, dtype=oracle.BF16, rope_theta=theta)
    kp = np.zeros((Pg, 1, 64, D), np.uint16)
    table = np.tile(np.arange(Pg, dtype=np.int32), (R, 1))
    kn = np.zeros((R, 1, D), np.uint16)
    q_out, rc = oracle.rope_write_kv(shape, qb, kn, kn.copy(), positions.astype(np.int32), table, kp, kp.copy())
    assert rc == 0
    C = f32(bf16_of(np.array([float(mpmath.cos(int(p))) for p in positions])))
    S = f32(bf16_of(np.array([float(mpmath.sin(int(p))) for p in positions])))
    want0 = bf16_of(C[:, None] * scales[None, :].astype(np.float64))
    # y_{D/2} = x_{D/2} * C + x_0 * S with x_{D/2} = 0 (so +0 at pos 0)
    want_h = bf16_of(0.0 * C[:, None] + S[:, None] * scales[None, :].astype(np.float64))
    assert np.array_equal(q_out[:, :, 0], want0)
    assert np.array_equal(q_out[:, :, D // 2], want_h)
