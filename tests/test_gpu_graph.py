"""The whole step captured in a CUDA graph and replayed.

A serving loop captures one decode step and replays it every token with the
inputs updated in place (positions advance, new q / k / v).  The replays
must match the oracle run step by step on the same inputs, and the planner
inside the graph must re-plan for the new positions.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_step_gb300 import workloads as wl

from gpu_util import binding, gpu_params, rope_tables_for, oracle_shape, assert_close

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


@pytest.mark.parametrize("chunk_pages", [0, 2])
def test_step_in_a_cuda_graph_replays_with_new_inputs(chunk_pages):
    b = binding()
    # positions keep pos % 64 < 63 so that pos + 1 stays in the row's last page
    w = wl.Workload("graph", rows=6, heads=32, kv_heads=8, head_dim=128, pages_per_row=12, dtype="bf16",
                    rope_theta=500000.0, positions="fixed", fixed_positions=(700, 0, 64, 130, 400, 765), seed=21)
    t = wl.generate(w, "cpu")
    host = {k: wl.to_numpy(v) for k, v in t.items()}
    d = {k: v.cuda() for k, v in t.items()}
    tables = rope_tables_for(b, w)
    p = gpu_params(b, w, host["k_pool"].shape[0], tables, chunk_pages)
    ws = b.new_workspace(p)
    out = torch.empty_like(d["q"])

    def step():
        b.decode_fused(p, d["q"], d["k_new"], d["v_new"], d["positions"], d["table"], d["k_pool"], d["v_pool"],
                       out, ws)

    # Eager warm-up on copies, so per-device set-up happens outside the capture.
    scratch = {k: v.clone() for k, v in d.items()}
    b.decode_fused(p, scratch["q"], scratch["k_new"], scratch["v_new"], scratch["positions"], scratch["table"],
                   scratch["k_pool"], scratch["v_pool"], torch.empty_like(out), ws)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()

    shape = oracle_shape(w, host["k_pool"].shape[0])
    kp, vp = host["k_pool"].copy(), host["v_pool"].copy()
    rng = torch.Generator().manual_seed(5)
    for it in range(3):
        graph.replay()
        torch.cuda.synchronize()
        b.check_status(ws)
        _, _, out64, rc = oracle.step(shape, host["q"], host["k_new"], host["v_new"], host["positions"],
                                      host["table"], kp, vp)
        assert rc == 0
        assert_close(out, out64, w.dtype, f"replay {it}")
        assert np.array_equal(wl.to_numpy(d["k_pool"]).view(np.uint8), kp.view(np.uint8))
        # next token: advance every row and draw new q / k / v, in place
        for name in ("q", "k_new", "v_new"):
            new = torch.randn(d[name].shape, generator=rng).to(w.torch_dtype)
            d[name].copy_(new)
            host[name] = wl.to_numpy(new)
        d["positions"].add_(1)
        host["positions"] = host["positions"] + 1


def test_prefill_and_packed_in_cuda_graphs():
    # Both calls issue three launches with no host synchronisation: they
    # capture as they are, and a replay picks up new inputs written in place.
    b = binding()
    rng = torch.Generator().manual_seed(9)

    # prefill: two rows, new tokens on cached prefixes
    w = wl.PrefillWorkload("graph_pf", prefix=(0, 90), chunk=(70, 40), heads=16, kv_heads=4, head_dim=128,
                           pages_per_row=3, rope_theta=500000.0, seed=22)
    t = wl.generate_prefill(w, "cpu")
    host = {k: wl.to_numpy(v) for k, v in t.items()}
    d = {k: v.cuda() for k, v in t.items()}
    cos, sin = b.rope_tables(w.rope_theta, w.head_dim, w.max_seq, torch.bfloat16)
    p = b.make_params(w.rows, w.heads, w.kv_heads, w.head_dim, w.pages_per_row, host["k_pool"].shape[0],
                      torch.bfloat16, rope_cos=cos, rope_sin=sin)
    ws = b.new_prefill_workspace(p, w.tokens)
    out = torch.empty_like(d["q"])
    names = ("q", "k_new", "v_new", "positions", "rows", "slots", "table", "k_pool", "v_pool")
    b.prefill_paged(p, *(d[k].clone() for k in names), torch.empty_like(out), ws)   # set-up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        b.prefill_paged(p, *(d[k] for k in names), out, ws)
    torch.cuda.synchronize()
    shape = oracle.make_shape(w.rows, w.heads, w.kv_heads, w.head_dim, w.pages_per_row, host["k_pool"].shape[0],
                              oracle.BF16, rope_theta=w.rope_theta)
    kp, vp = host["k_pool"].copy(), host["v_pool"].copy()
    for it in range(2):
        graph.replay()
        torch.cuda.synchronize()
        b.check_status(ws)
        _, _, out64, rc = oracle.prefill_paged(shape, host["q"], host["k_new"], host["v_new"], host["positions"],
                                               host["rows"], host["slots"], host["table"], kp, vp)
        assert rc == 0
        assert_close(out, out64, "bf16", f"prefill replay {it}")
        assert np.array_equal(wl.to_numpy(d["k_pool"]).view(np.uint8), kp.view(np.uint8))
        for name in ("q", "k_new", "v_new"):
            new = torch.randn(d[name].shape, generator=rng).to(torch.bfloat16)
            d[name].copy_(new)
            host[name] = wl.to_numpy(new)

    # packed: three sequences in one row
    w = wl.PackedWorkload("graph_pk", lengths=(100, 37, 64), heads=16, kv_heads=4, head_dim=64, seed=23)
    t = wl.generate_packed(w, "cpu")
    host = {k: wl.to_numpy(v) for k, v in t.items()}
    d = {k: v.cuda() for k, v in t.items()}
    cos, sin = b.rope_tables(w.rope_theta, w.head_dim, w.max_seq, torch.bfloat16)
    p = b.make_params(1, w.heads, w.kv_heads, w.head_dim, 1, 1, torch.bfloat16, rope_cos=cos, rope_sin=sin)
    ws = b.new_packed_workspace(p, w.tokens)
    out = torch.empty_like(d["q"])
    names = ("q", "k", "v", "positions", "segments")
    b.packed(p, *(d[k].clone() for k in names), torch.empty_like(out), ws)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        b.packed(p, *(d[k] for k in names), out, ws)
    torch.cuda.synchronize()
    shape = oracle.make_shape(0, w.heads, w.kv_heads, w.head_dim, 1, 1, oracle.BF16, rope_theta=w.rope_theta)
    for it in range(2):
        graph.replay()
        torch.cuda.synchronize()
        b.check_status(ws)
        _, _, _, out64, rc = oracle.packed(shape, host["q"], host["k"], host["v"], host["positions"],
                                           host["segments"])
        assert rc == 0
        assert_close(out, out64, "bf16", f"packed replay {it}")
        for name in ("q", "k", "v"):
            new = torch.randn(d[name].shape, generator=rng).to(torch.bfloat16)
            d[name].copy_(new)
            host[name] = wl.to_numpy(new)
