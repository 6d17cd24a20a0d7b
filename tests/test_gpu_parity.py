"""GPU parity: the CUDA path (through the C-ABI) against the CPU oracle.

Cache writes and rotated queries must match bit for bit; attention outputs
within max |err| <= 2e-2 and mean |err| <= 2e-3 of the fp64 oracle for bf16,
1e-5 for f32.
"""
import os
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_step_gb300 import workloads as wl

from gpu_util import binding, run_step, rope_tables_for, gpu_params, oracle_shape, assert_close

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


def W(name="t", R=4, Hq=32, Hk=8, D=128, Pg=6, dtype="bf16", theta=500000.0, window=0, positions=None,
      num_pages=0, seed=7):
    if positions is None:
        positions = tuple(int(x) for x in np.random.default_rng(seed).integers(0, Pg * 64, R))
    return wl.Workload(name, rows=len(positions), heads=Hq, kv_heads=Hk, head_dim=D, pages_per_row=Pg,
                       dtype=dtype, rope_theta=theta, window=window, positions="fixed",
                       fixed_positions=tuple(positions), num_pages=num_pages, seed=seed)


# ---------------------------------------------------------------- tables ----
@pytest.mark.parametrize("theta,D,S,dtype", [(10000.0, 64, 512, torch.bfloat16),
                                              (500000.0, 128, 8192, torch.bfloat16),
                                              (150000.0, 64, 4096, torch.bfloat16),
                                              (500000.0, 128, 2048, torch.float32)])
def test_rope_tables_bit_exact(theta, D, S, dtype):
    b = binding()
    cos, sin = b.rope_tables(theta, D, S, dtype)
    od = oracle.BF16 if dtype == torch.bfloat16 else oracle.F32
    c, s = oracle.rope_tables(theta, D, S, od)
    assert np.array_equal(wl.to_numpy(cos).view(np.uint8), c.view(np.uint8))
    assert np.array_equal(wl.to_numpy(sin).view(np.uint8), s.view(np.uint8))


# ------------------------------------------------------------ the step ------
def test_tiny_workload():
    run_step(wl.TINY)


@pytest.mark.parametrize("mode", ["fused", "split"])
def test_llama_shape_small(mode):
    run_step(W(positions=(0, 1, 63, 64, 65, 127, 128, 383, 200, 5)), mode=mode)


@pytest.mark.parametrize("Hq,Hk,D", [(8, 8, 64), (16, 8, 64), (32, 8, 64), (64, 8, 64), (8, 8, 128),
                                     (16, 8, 128), (64, 8, 128), (12, 12, 64), (7, 1, 128)])
def test_group_sizes_and_head_dims(Hq, Hk, D):
    run_step(W(Hq=Hq, Hk=Hk, D=D, Pg=5, positions=(0, 64, 100, 319, 250), theta=10000.0, seed=Hq * D))


@pytest.mark.parametrize("window", [1, 2, 63, 64, 65, 128, 300])
def test_sliding_window(window):
    run_step(W(Hq=64, Hk=8, D=64, Pg=8, window=window, theta=150000.0,
               positions=(0, 5, 63, 64, 127, 128, 129, 511, 300, 200)), poison=True)


@pytest.mark.parametrize("chunk_pages", [1, 2, 3, 5])
def test_forced_splits_merge(chunk_pages):
    run_step(W(R=6, Pg=12, positions=(767, 700, 64, 0, 400, 130)), chunk_pages=chunk_pages)


@pytest.mark.parametrize("chunk_pages", [0, 1, 3])
def test_unreadable_slots_hold_nan(chunk_pages):
    run_step(W(R=5, Pg=6, positions=(0, 70, 191, 383, 32), num_pages=40), poison=True, chunk_pages=chunk_pages)


@pytest.mark.parametrize("Hq,Hk,D,window", [(12, 12, 64, 0), (12, 12, 64, 100), (32, 8, 128, 0), (8, 1, 64, 0)])
def test_f32(Hq, Hk, D, window):
    run_step(W(Hq=Hq, Hk=Hk, D=D, dtype="f32", theta=0.0, Pg=6, window=window,
               positions=(0, 1, 64, 65, 383, 255)), poison=True)
    run_step(W(Hq=Hq, Hk=Hk, D=D, dtype="f32", theta=0.0, Pg=6, window=window,
               positions=(0, 1, 64, 65, 383, 255)), chunk_pages=2)


def test_f32_with_rope():
    run_step(W(Hq=16, Hk=4, D=128, dtype="f32", theta=10000.0, Pg=4, positions=(3, 200, 255)))


def test_maximum_position_and_single_row():
    run_step(W(R=1, Pg=128, positions=(8191,), theta=500000.0))
    run_step(W(R=1, Pg=2, positions=(127,), Hq=8, Hk=8, D=64, theta=10000.0), chunk_pages=1)


def test_many_rows_short_contexts():
    rng = np.random.default_rng(5)
    run_step(W(R=300, Pg=2, Hq=8, Hk=2, D=64, theta=10000.0, positions=tuple(int(x) for x in rng.integers(0, 128, 300))))


@pytest.mark.parametrize("chunk_pages", [0, 1])
def test_more_rows_than_the_planner_block(chunk_pages):
    # 700 rows take the planner's general path (more rows than threads)
    rng = np.random.default_rng(6)
    run_step(W(R=700, Pg=3, Hq=8, Hk=2, D=64, theta=10000.0,
               positions=tuple(int(x) for x in rng.integers(0, 192, 700))), chunk_pages=chunk_pages)


# ----------------------------------------------------- attention sinks -----
@pytest.mark.parametrize("window,chunk_pages", [(0, 0), (128, 0), (0, 2), (100, 1)])
def test_attention_sinks_gptoss_shape(window, chunk_pages):
    # gpt-oss-20b page, SinkAttention `param sinks: Tensor[Heads; T]`
    rng = np.random.default_rng(window + chunk_pages)
    sinks = rng.standard_normal(64).tolist()
    run_step(W(Hq=64, Hk=8, D=64, Pg=8, window=window, theta=150000.0,
               positions=(0, 5, 63, 64, 200, 511, 300)), chunk_pages=chunk_pages, sinks=sinks)


def test_attention_sinks_extreme_values_and_f32():
    sinks = [12.0, -12.0, 0.0, 3.0] * 4
    run_step(W(Hq=16, Hk=4, D=128, Pg=4, positions=(0, 100, 255), theta=10000.0), sinks=sinks)
    run_step(W(Hq=16, Hk=4, D=64, dtype="f32", theta=0.0, Pg=4, positions=(0, 100, 255)), sinks=sinks,
             chunk_pages=1)


# ------------------------------------------------------- repeat / reuse -----
def test_attend_twice_on_one_plan_is_identical():
    b = binding()
    w = W(R=6, Pg=12, positions=(767, 700, 64, 0, 400, 130))
    t = {k: v.cuda() for k, v in wl.generate(w, "cpu").items()}
    tables = rope_tables_for(b, w)
    p = gpu_params(b, w, t["k_pool"].shape[0], tables, chunk_pages=2)
    ws = b.new_workspace(p)
    q_rot = torch.empty_like(t["q"])
    b.rope_write_kv(p, t["q"], t["k_new"], t["v_new"], t["positions"], t["table"], q_rot, t["k_pool"],
                    t["v_pool"], ws)
    b.plan(p, t["positions"], ws)
    outs = []
    for _ in range(3):
        out = torch.full_like(t["q"], float("nan"))
        b.attend(p, q_rot, t["positions"], t["table"], t["k_pool"], t["v_pool"], out, ws)
        outs.append(out)
    b.check_status(ws)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


def test_q_out_may_alias_q():
    b = binding()
    w = W(R=3, Pg=3, positions=(10, 100, 190), Hq=16, Hk=4, D=64, theta=10000.0)
    t = {k: v.cuda() for k, v in wl.generate(w, "cpu").items()}
    tables = rope_tables_for(b, w)
    p = gpu_params(b, w, t["k_pool"].shape[0], tables)
    ws = b.new_workspace(p)
    sep = torch.empty_like(t["q"])
    b.rope_write_kv(p, t["q"], t["k_new"], t["v_new"], t["positions"], t["table"], sep, t["k_pool"],
                    t["v_pool"], ws)
    q = t["q"].clone()
    b.rope_write_kv(p, q, t["k_new"], t["v_new"], t["positions"], t["table"], q, t["k_pool"], t["v_pool"], ws)
    b.check_status(ws)
    assert torch.equal(q.view(torch.int16), sep.view(torch.int16))


# ------------------------------------------------------ device errors -------
def _setup(w, chunk_pages=0):
    b = binding()
    t = {k: v.cuda() for k, v in wl.generate(w, "cpu").items()}
    tables = rope_tables_for(b, w)
    p = gpu_params(b, w, t["k_pool"].shape[0], tables, chunk_pages)
    return b, t, p, b.new_workspace(p)


def test_bad_page_id_reports_error_and_spares_other_rows():
    w = W(R=3, Pg=4, positions=(100, 200, 30))
    b, t, p, ws = _setup(w)
    t["table"][1, 1] = 10 ** 6
    out = torch.zeros_like(t["q"])
    b.decode_fused(p, t["q"], t["k_new"], t["v_new"], t["positions"], t["table"], t["k_pool"], t["v_pool"], out, ws)
    with pytest.raises(b.PdattnError) as e:
        b.check_status(ws)
    assert e.value.status == b.EBADPAGE
    b.check_status(ws)                   # cleared


def test_bad_position_reports_error():
    w = W(R=2, Pg=4, positions=(100, 200))
    b, t, p, ws = _setup(w)
    t["positions"][0] = 4 * 64          # one past the table
    out = torch.zeros_like(t["q"])
    b.decode_fused(p, t["q"], t["k_new"], t["v_new"], t["positions"], t["table"], t["k_pool"], t["v_pool"], out, ws)
    with pytest.raises(b.PdattnError) as e:
        b.check_status(ws)
    assert e.value.status == b.EBADPOS


def test_attend_without_plan_is_refused_on_device():
    w = W(R=2, Pg=4, positions=(100, 200))
    b, t, p, ws = _setup(w)
    out = torch.zeros_like(t["q"])
    b.attend(p, t["q"], t["positions"], t["table"], t["k_pool"], t["v_pool"], out, ws)
    with pytest.raises(b.PdattnError) as e:
        b.check_status(ws)
    assert e.value.status == b.EINVAL


# ------------------------------------------------- full-size workloads ------
FULL = [wl.LLAMA_LAYER, wl.LLAMA_SERVING, wl.GPTOSS_FULL, wl.GPTOSS_SLIDING, wl.GPT2]


@pytest.mark.parametrize("w", FULL, ids=[w.name for w in FULL])
def test_full_size_whole_batch(w):
    """The bench's launch (decode_fused, planner's split choice) at full size;
    the oracle recomputes every row (its rows on all host cores) and both
    pools are compared whole, bit for bit."""
    b = binding()
    t = wl.generate(w, "cuda")
    host = {k: wl.to_numpy(v) for k, v in t.items()}
    num_pages = host["k_pool"].shape[0]
    tables = rope_tables_for(b, w)
    p = gpu_params(b, w, num_pages, tables)
    ws = b.new_workspace(p)
    out = torch.empty_like(t["q"])
    b.decode_fused(p, t["q"], t["k_new"], t["v_new"], t["positions"], t["table"], t["k_pool"], t["v_pool"], out, ws)
    b.check_status(ws)
    kp, vp = host["k_pool"], host["v_pool"]
    oracle.set_threads(os.cpu_count() or 1)
    try:
        _, _, out64, rc = oracle.step(oracle_shape(w, num_pages), host["q"], host["k_new"], host["v_new"],
                                      host["positions"], host["table"], kp, vp)
    finally:
        oracle.set_threads(1)
    assert rc == 0
    assert_close(out, out64, w.dtype, w.name)
    assert np.array_equal(wl.to_numpy(t["k_pool"]).view(np.uint8), kp.view(np.uint8)), "k pool differs"
    assert np.array_equal(wl.to_numpy(t["v_pool"]).view(np.uint8), vp.view(np.uint8)), "v pool differs"


@pytest.mark.parametrize("mode", ["fused", "layers"])
def test_decode_loop_with_advancing_positions(mode):
    """A serving loop: ten steps on one workspace, each row's position one
    further every step (crossing page boundaries), new q / k / v each step.
    Every step's output is checked against the oracle, which runs the same
    steps on its own copy of the pools; the pools are compared at the end."""
    b = binding()
    R, steps = 48, 10
    rng = np.random.default_rng(21)
    start = rng.integers(0, 6 * 64 - steps, R)
    start[:6] = [54, 55, 62, 63, 118, 0]               # rows that cross page boundaries
    w = W("loop", R=R, Pg=6, Hq=32, Hk=8, D=128, positions=tuple(int(x) for x in start + steps - 1), seed=21)
    t = wl.generate(w, "cpu")
    host = {k: wl.to_numpy(v) for k, v in t.items()}
    kp, vp = host["k_pool"].copy(), host["v_pool"].copy()
    num_pages = kp.shape[0]
    shape = oracle_shape(w, num_pages)
    tables = rope_tables_for(b, w)
    p = gpu_params(b, w, num_pages, tables)
    d = {k: v.cuda() for k, v in t.items()}
    ws = b.new_layers_workspace(p, 1) if mode == "layers" else b.new_workspace(p)
    gen = torch.Generator().manual_seed(22)
    for s in range(steps):
        pos = torch.tensor(start + s, dtype=torch.int32)
        q = torch.randn(R, w.heads, w.head_dim, generator=gen).to(torch.bfloat16)
        kn = torch.randn(R, w.kv_heads, w.head_dim, generator=gen).to(torch.bfloat16)
        vn = torch.randn(R, w.kv_heads, w.head_dim, generator=gen).to(torch.bfloat16)
        _, _, out64, rc = oracle.step(shape, wl.to_numpy(q), wl.to_numpy(kn), wl.to_numpy(vn), wl.to_numpy(pos),
                                      host["table"], kp, vp)
        assert rc == 0
        out = torch.full((R, w.heads, w.head_dim), float("nan"), dtype=torch.bfloat16, device="cuda")
        if mode == "fused":
            b.decode_fused(p, q.cuda(), kn.cuda(), vn.cuda(), pos.cuda(), d["table"], d["k_pool"], d["v_pool"], out, ws)
        else:
            b.decode_layers(p, [dict(q=q.cuda(), k_new=kn.cuda(), v_new=vn.cuda(), k_pool=d["k_pool"],
                                     v_pool=d["v_pool"], out=out)], pos.cuda(), d["table"], ws)
        b.check_status(ws)
        assert_close(out, out64, "bf16", f"step {s}")
    assert np.array_equal(wl.to_numpy(d["k_pool"]).view(np.uint8), kp.view(np.uint8))
    assert np.array_equal(wl.to_numpy(d["v_pool"]).view(np.uint8), vp.view(np.uint8))
