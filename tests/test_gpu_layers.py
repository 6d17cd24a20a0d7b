"""Several layers' decode steps in one group of launches (pdattn_decode_layers)
against the oracle run layer by layer.

Every layer has its own q, new k and v, pools, window and sinks; positions
and the page table are shared (the model pages repeat one decoder layer, and
the gpt-oss-20b page alternates a sliding-window and a full layer in each
`LayerPair`).  Each layer's output must match the oracle within the bf16
(f32) tolerance and each layer's pools bit for bit.
"""
import os
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_step_gb300 import workloads as wl

from gpu_util import binding, gpu_params, oracle_shape, rope_tables_for, assert_close

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


def make_layers(w, n_layers, windows, sink_heads=None, seed=0):
    """Shared positions and table from the workload's draw; per layer fresh
    N(0, 1) q, k_new, v_new and pools of the same shapes (host numpy)."""
    base = {k: wl.to_numpy(v) for k, v in wl.generate(w, "cpu").items()}
    gen = torch.Generator().manual_seed(10_000 + seed)
    layers = []
    for l in range(n_layers):
        y = {}
        for k in ("q", "k_new", "v_new", "k_pool", "v_pool"):
            x = torch.randn(*base[k].shape, generator=gen, dtype=torch.float32).to(w.torch_dtype)
            y[k] = wl.to_numpy(x)
        y["window"] = windows[l % len(windows)]
        y["sinks"] = None
        if sink_heads is not None and l % 2 == 0:
            s = (torch.randn(w.heads, generator=gen) * 2.0).to(w.torch_dtype)
            y["sinks"] = wl.to_numpy(s)
        layers.append(y)
    return base, layers


def oracle_layers(w, base, layers):
    """Per layer: rope + write into copies of its pools, then attention with
    its window and sinks.  Returns [(out64, k_pool, v_pool)]."""
    res = []
    oracle.set_threads(os.cpu_count() or 1)
    try:
        for y in layers:
            shape = oracle_shape(replace(w, window=y["window"]), y["k_pool"].shape[0])
            kp, vp = y["k_pool"].copy(), y["v_pool"].copy()
            q_rot, rc = oracle.rope_write_kv(shape, y["q"], y["k_new"], y["v_new"], base["positions"], base["table"],
                                             kp, vp)
            assert rc == 0
            _, out64, rc = oracle.decode(shape, q_rot, base["positions"], base["table"], kp, vp, y["sinks"])
            assert rc == 0
            res.append((out64, kp, vp))
    finally:
        oracle.set_threads(1)
    return res


def run_layers(w, n_layers, windows, sink_heads=None, seed=0, repeat=1):
    b = binding()
    base, layers = make_layers(w, n_layers, windows, sink_heads, seed)
    want = oracle_layers(w, base, layers)
    dt = w.torch_dtype
    dev = lambda a: wl.from_numpy(a, dt).cuda() if a.dtype != np.int32 else torch.from_numpy(a.copy()).cuda()
    num_pages = base["k_pool"].shape[0]
    p = gpu_params(b, w, num_pages, rope_tables_for(b, w))
    ws = b.new_layers_workspace(p, n_layers)
    d_layers = []
    for y in layers:
        d = {k: dev(y[k]) for k in ("q", "k_new", "v_new", "k_pool", "v_pool")}
        d["out"] = torch.full_like(d["q"], float("nan"))
        d["window"] = y["window"]
        d["sinks"] = None if y["sinks"] is None else dev(y["sinks"])
        d_layers.append(d)
    positions, table = dev(base["positions"]), dev(base["table"])
    for _ in range(repeat):
        b.decode_layers(p, d_layers, positions, table, ws)
        b.check_status(ws)
        assert b.last_launch_count() == 3 * ((n_layers + b.LAYERS_PER_LAUNCH - 1) // b.LAYERS_PER_LAUNCH)
    for l, (d, (out64, kp, vp)) in enumerate(zip(d_layers, want)):
        assert_close(d["out"], out64, w.dtype, f"layer {l}")
        assert np.array_equal(wl.to_numpy(d["k_pool"]).view(np.uint8), kp.view(np.uint8)), f"layer {l} k pool"
        assert np.array_equal(wl.to_numpy(d["v_pool"]).view(np.uint8), vp.view(np.uint8)), f"layer {l} v pool"


SMALL_GPTOSS = wl.Workload("pair", rows=12, heads=64, kv_heads=8, head_dim=64, pages_per_row=20, dtype="bf16",
                           rope_theta=150000.0, positions="uniform", pos_lo=0, pos_hi=1279, seed=51)


def test_layer_pair_sliding_and_full_with_sinks():
    # gpt-oss-20b LayerPair: a window-128 layer with sinks, then a full layer
    run_layers(SMALL_GPTOSS, 2, windows=(128, 0), sink_heads=True, seed=1)


def test_twelve_layers_alternating_called_twice():
    run_layers(SMALL_GPTOSS, 12, windows=(128, 0, 1, 300), sink_heads=True, seed=2, repeat=2)


def test_more_layers_than_one_launch_serves():
    # 35 layers: a group of launches for 32, then one for 3, on the same workspace
    w = wl.Workload("many", rows=3, heads=32, kv_heads=8, head_dim=128, pages_per_row=4, dtype="bf16",
                    rope_theta=500000.0, positions="fixed", fixed_positions=(0, 130, 255), seed=52)
    run_layers(w, 35, windows=(0, 64), seed=3)


def test_gpt2_f32_layers():
    w = wl.Workload("gpt2_layers", rows=10, heads=12, kv_heads=12, head_dim=64, pages_per_row=16, dtype="f32",
                    rope_theta=0.0, positions="uniform", pos_lo=1, pos_hi=1023, seed=53)
    run_layers(w, 3, windows=(0,), seed=4)


def test_llama_layers_with_groups_of_four():
    w = wl.Workload("llama_layers", rows=20, heads=32, kv_heads=8, head_dim=128, pages_per_row=32, dtype="bf16",
                    rope_theta=500000.0, positions="loguniform_ctx", pos_lo=16, pos_hi=2048, seed=54)
    run_layers(w, 4, windows=(0,), seed=5)


def test_full_size_gptoss_layer_pair():
    # the gpt-oss-20b shape at full size (64 rows, positions up to 4095):
    # both layers of the pair, every row
    run_layers(wl.GPTOSS_FULL, 2, windows=(128, 0), sink_heads=True, seed=6)


def test_layers_beyond_the_first_wave_rows():
    # 6 layers x 100 rows = 600 launch rows: more than the planner's one-row-
    # per-thread path takes, so the general planner runs and no CTA starts early
    w = wl.Workload("wide", rows=100, heads=16, kv_heads=4, head_dim=64, pages_per_row=4, dtype="bf16",
                    rope_theta=10000.0, positions="uniform", pos_lo=0, pos_hi=255, seed=55)
    run_layers(w, 6, windows=(0, 100, 7), sink_heads=True, seed=7, repeat=2)
