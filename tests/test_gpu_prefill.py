"""Paged prefill on the GPU against the oracle.

The CUDA path (rope + write at slots, tile list, tensor-core attention)
through the C-ABI, and the oracle's prefill on the same seeded inputs: the
pools must match bit for bit, the outputs within the bf16 tolerance.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_step_gb300 import workloads as wl

from gpu_util import binding, assert_close

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


def inputs(w, q_scale=1.0, poison=False, permute=False):
    t = wl.generate_prefill(w, "cpu")
    if q_scale != 1.0:
        t["q"] = (t["q"].float() * q_scale).to(w.torch_dtype)     # power of two: exact
    a = {k: wl.to_numpy(v) for k, v in t.items()}
    if poison:
        # slots past each row's last new token hold no key yet: NaN must not leak
        nan = oracle.f32_to_bf16_bits(float("nan"))
        for r, (p0, c) in enumerate(zip(w.prefix, w.chunk)):
            end = p0 + c
            page = a["table"][r, (end - 1) // 64]
            a["k_pool"][page, :, (end - 1) % 64 + 1:, :] = nan
            a["v_pool"][page, :, (end - 1) % 64 + 1:, :] = nan
    if permute:
        order = np.random.default_rng(w.seed).permutation(w.tokens)
        for k in ("q", "k_new", "v_new", "positions", "rows", "slots"):
            a[k] = np.ascontiguousarray(a[k][order])
    return a


def to_dev(a):
    return {k: wl.from_numpy(v, torch.bfloat16 if v.dtype == np.uint16 else torch.int32).cuda()
            for k, v in a.items()}


def out_like(q, misalign):
    # misalign: an output 16 but not 32 bytes aligned (the epilogue's narrow stores)
    if not misalign:
        return torch.empty_like(q)
    flat = torch.empty(q.numel() + 16, dtype=q.dtype, device=q.device)
    base = flat.data_ptr() % 32 // 2                 # elements past a 32-byte boundary
    o = flat[(8 - base) % 16: (8 - base) % 16 + q.numel()].view(q.shape)
    assert o.data_ptr() % 32 == 16
    return o


def run(w, sinks=None, misalign=False, **kw):
    b = binding()
    a = inputs(w, **kw)
    num_pages = a["k_pool"].shape[0]
    shape = oracle.make_shape(w.rows, w.heads, w.kv_heads, w.head_dim, w.pages_per_row, num_pages, oracle.BF16,
                              window=w.window, rope_theta=w.rope_theta)
    sink_t = None if sinks is None else torch.tensor(sinks, dtype=torch.float32).to(torch.bfloat16)
    kp, vp = a["k_pool"].copy(), a["v_pool"].copy()
    _, _, out64, rc = oracle.prefill_paged(shape, a["q"], a["k_new"], a["v_new"], a["positions"], a["rows"],
                                           a["slots"], a["table"], kp, vp,
                                           None if sink_t is None else wl.to_numpy(sink_t))
    assert rc == 0
    d = to_dev(a)
    cos, sin = b.rope_tables(w.rope_theta, w.head_dim, w.max_seq, torch.bfloat16)
    p = b.make_params(w.rows, w.heads, w.kv_heads, w.head_dim, w.pages_per_row, num_pages, torch.bfloat16,
                      window=w.window, rope_cos=cos, rope_sin=sin,
                      sinks=None if sink_t is None else sink_t.cuda())
    ws = b.new_prefill_workspace(p, w.tokens)
    out = out_like(d["q"], misalign)
    b.prefill_paged(p, d["q"], d["k_new"], d["v_new"], d["positions"], d["rows"], d["slots"], d["table"],
                    d["k_pool"], d["v_pool"], out, ws)
    b.check_status(ws)
    assert b.last_launch_count() == 3
    assert np.array_equal(wl.to_numpy(d["k_pool"]).view(np.uint8), kp.view(np.uint8)), "k pool differs"
    assert np.array_equal(wl.to_numpy(d["v_pool"]).view(np.uint8), vp.view(np.uint8)), "v pool differs"
    err = assert_close(out, out64, "bf16", w.name)
    print(f"{w.name}: max |err| {err[0]:.4g}, mean |err| {err[1]:.3g}")
    return err


def W(name, prefix, chunk, heads, kv_heads, head_dim, **kw):
    pages = max((p + c + 63) // 64 for p, c in zip(prefix, chunk)) + kw.pop("extra_pages", 1)
    return wl.PrefillWorkload(name, prefix=tuple(prefix), chunk=tuple(chunk), heads=heads, kv_heads=kv_heads,
                              head_dim=head_dim, pages_per_row=pages, **kw)


def test_prefill_small_ragged_tiles():
    run(W("small", (0, 70, 5), (40, 30, 64), 8, 2, 64, seed=1))


@pytest.mark.parametrize("heads,kv_heads,head_dim", [
    (4, 4, 64), (4, 4, 128), (8, 4, 64), (8, 4, 128), (16, 4, 64), (16, 4, 128), (16, 2, 64), (16, 2, 128),
    (6, 2, 64), (12, 2, 128),              # g = 3, 6: tiles of 42 / 21 tokens, spare MMA rows
])
def test_prefill_groups_and_head_dims(heads, kv_heads, head_dim):
    run(W(f"g{heads // kv_heads}d{head_dim}", (0, 130, 64), (150, 77, 1), heads, kv_heads, head_dim,
          rope_theta=500000.0, seed=2))


def test_prefill_llama_shape():
    run(W("llama", (0, 1000, 300), (300, 100, 257), 32, 8, 128, rope_theta=500000.0, seed=3))


@pytest.mark.parametrize("head_dim", [64, 128])
def test_prefill_output_aligned_to_16_bytes_only(head_dim):
    run(W("misaligned", (0, 200), (130, 70), 16, 4, head_dim, rope_theta=500000.0, seed=13), misalign=True)


@pytest.mark.parametrize("window", [1, 64, 128, 200])
def test_prefill_sliding_window(window):
    run(W("window", (0, 400, 60), (260, 90, 70), 64, 8, 64, rope_theta=150000.0, window=window, seed=4))


def test_prefill_sinks_gpt_oss_shape():
    sinks = list(np.random.default_rng(5).normal(0.0, 2.0, 64))
    run(W("sinks", (0, 300), (200, 129), 64, 8, 64, rope_theta=150000.0, window=128, seed=5), sinks=sinks)


def test_prefill_large_logits_rescale_path():
    # q scaled by 16: logits spread over many powers of two, so the running
    # max often grows past the lazy-rescale threshold
    run(W("rescale", (0, 500), (700, 300), 32, 8, 128, rope_theta=500000.0, seed=6), q_scale=16.0)


def test_prefill_nan_in_unwritten_slots_does_not_leak():
    run(W("poison", (0, 70, 5), (40, 30, 64), 8, 2, 128, seed=7), poison=True)


def test_prefill_tokens_in_any_order():
    run(W("permuted", (0, 100, 30), (120, 64, 50), 16, 4, 64, seed=8), permute=True)


def test_prefill_one_token_per_row_matches_decode_step():
    run(W("decode_like", (63, 700, 0, 128), (1, 1, 1, 1), 32, 8, 128, rope_theta=500000.0, seed=9))


def test_prefill_full_size_sampled_tokens():
    # Llama-3.1-8B shape, 8 rows x 1024 new tokens on prefixes 0 .. 7168.
    # The oracle writes every token (as rows of a decode write) and attends
    # a sample of tokens, each as a one-row decode over its table row.
    b = binding()
    w = wl.PREFILL_LLAMA
    a = inputs(w)
    num_pages = a["k_pool"].shape[0]
    P = w.tokens
    tab_tok = np.ascontiguousarray(a["table"][a["rows"]])
    shape_tok = oracle.make_shape(P, w.heads, w.kv_heads, w.head_dim, w.pages_per_row, num_pages, oracle.BF16,
                                  rope_theta=w.rope_theta)
    kp, vp = a["k_pool"].copy(), a["v_pool"].copy()
    q_rot, rc = oracle.rope_write_kv(shape_tok, a["q"], a["k_new"], a["v_new"], a["positions"], tab_tok, kp, vp)
    assert rc == 0
    d = to_dev(a)
    cos, sin = b.rope_tables(w.rope_theta, w.head_dim, w.max_seq, torch.bfloat16)
    p = b.make_params(w.rows, w.heads, w.kv_heads, w.head_dim, w.pages_per_row, num_pages, torch.bfloat16,
                      rope_cos=cos, rope_sin=sin)
    ws = b.new_prefill_workspace(p, P)
    out = torch.empty_like(d["q"])
    b.prefill_paged(p, d["q"], d["k_new"], d["v_new"], d["positions"], d["rows"], d["slots"], d["table"],
                    d["k_pool"], d["v_pool"], out, ws)
    b.check_status(ws)
    assert np.array_equal(wl.to_numpy(d["k_pool"]).view(np.uint8), kp.view(np.uint8))
    assert np.array_equal(wl.to_numpy(d["v_pool"]).view(np.uint8), vp.view(np.uint8))
    got = out.cpu()
    # every token of two whole rows, the longest prefix and a middle one,
    # each token a decode row of the oracle (its rows on all host cores)
    rows = [w.rows - 1, w.rows // 2 - 1]
    idx = np.flatnonzero(np.isin(a["rows"], rows))
    shape = oracle.make_shape(len(idx), w.heads, w.kv_heads, w.head_dim, w.pages_per_row, num_pages, oracle.BF16)
    oracle.set_threads(os.cpu_count() or 1)
    try:
        _, o64, rc = oracle.decode(shape, np.ascontiguousarray(q_rot[idx]), np.ascontiguousarray(a["positions"][idx]),
                                   np.ascontiguousarray(tab_tok[idx]), kp, vp)
    finally:
        oracle.set_threads(1)
    assert rc == 0
    assert_close(got[torch.as_tensor(idx)], o64, "bf16", f"rows {rows}")


def test_prefill_attend_reruns_the_attention_bit_for_bit():
    # 26 tiles x 8 kv heads = 208 units on at most 152 CTAs: CTAs take units
    # from the cursor, which the last CTA out must rewind for the next launch
    b = binding()
    w = W("again", (0, 200), (900, 700), 32, 8, 128, rope_theta=500000.0, seed=10)
    d = to_dev(inputs(w))
    cos, sin = b.rope_tables(w.rope_theta, w.head_dim, w.max_seq, torch.bfloat16)
    p = b.make_params(w.rows, w.heads, w.kv_heads, w.head_dim, w.pages_per_row, d["k_pool"].shape[0],
                      torch.bfloat16, rope_cos=cos, rope_sin=sin)
    ws = b.new_prefill_workspace(p, w.tokens)
    out1, out2 = torch.empty_like(d["q"]), torch.full_like(d["q"], float("nan"))
    b.prefill_paged(p, d["q"], d["k_new"], d["v_new"], d["positions"], d["rows"], d["slots"], d["table"],
                    d["k_pool"], d["v_pool"], out1, ws)
    for _ in range(3):
        out2.fill_(float("nan"))
        b.prefill_attend(p, d["positions"], d["table"], d["k_pool"], d["v_pool"], out2, ws)
        b.check_status(ws)
        assert b.last_launch_count() == 1
        assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
