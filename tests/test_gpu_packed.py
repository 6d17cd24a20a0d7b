"""Packed sequences on the GPU against the oracle.

The CUDA path (tile planner, rope of q and k, tensor-core attention over the
pack's 64-token key blocks) through the C-ABI, and the oracle's packed
attention on the same seeded inputs, outputs within the bf16 tolerance.
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


def to_dev(a):
    return {k: wl.from_numpy(v, torch.bfloat16 if v.dtype == np.uint16 else torch.int32).cuda()
            for k, v in a.items()}


def gpu_packed(w, a, sinks_t=None, misalign=False):
    b = binding()
    d = to_dev(a)
    cos, sin = b.rope_tables(w.rope_theta, w.head_dim, int(a["positions"].max()) + 1, torch.bfloat16)
    # rows / pages / pool fields are not read by the packed entry
    p = b.make_params(1, w.heads, w.kv_heads, w.head_dim, 1, 1, torch.bfloat16, window=w.window, rope_cos=cos,
                      rope_sin=sin, sinks=sinks_t)
    ws = b.new_packed_workspace(p, len(a["positions"]))
    if misalign:
        # an output 16 but not 32 bytes aligned (the epilogue's narrow stores)
        flat = torch.empty(d["q"].numel() + 16, dtype=d["q"].dtype, device=d["q"].device)
        off = (8 - flat.data_ptr() % 32 // 2) % 16
        out = flat[off:off + d["q"].numel()].view(d["q"].shape)
        assert out.data_ptr() % 32 == 16
    else:
        out = torch.empty_like(d["q"])
    b.packed(p, d["q"], d["k"], d["v"], d["positions"], d["segments"], out, ws)
    b.check_status(ws)
    assert b.last_launch_count() == 3
    return out


def run(w, sinks=None, q_scale=1.0, transform=None, misalign=False):
    t = wl.generate_packed(w, "cpu")
    if q_scale != 1.0:
        t["q"] = (t["q"].float() * q_scale).to(torch.bfloat16)
    a = {k: wl.to_numpy(v) for k, v in t.items()}
    if transform is not None:
        a = transform(a)
    shape = oracle.make_shape(0, w.heads, w.kv_heads, w.head_dim, 1, 1, oracle.BF16, window=w.window,
                              rope_theta=w.rope_theta)
    sink_t = None if sinks is None else torch.tensor(sinks, dtype=torch.float32).to(torch.bfloat16)
    _, _, _, out64, rc = oracle.packed(shape, a["q"], a["k"], a["v"], a["positions"], a["segments"],
                                       None if sink_t is None else wl.to_numpy(sink_t))
    assert rc == 0
    out = gpu_packed(w, a, None if sink_t is None else sink_t.cuda(), misalign)
    err = assert_close(out, out64, "bf16", w.name)
    print(f"{w.name}: max |err| {err[0]:.4g}, mean |err| {err[1]:.3g}")


def W(name, lengths, heads, kv_heads, head_dim, **kw):
    return wl.PackedWorkload(name, lengths=tuple(lengths), heads=heads, kv_heads=kv_heads, head_dim=head_dim, **kw)


def test_packed_small_ragged():
    run(W("small", (40, 70, 5, 130), 8, 2, 64, seed=1))


@pytest.mark.parametrize("head_dim", [64, 128])
def test_packed_output_aligned_to_16_bytes_only(head_dim):
    run(W("misaligned", (100, 33, 180), 16, 4, head_dim, rope_theta=500000.0, seed=14), misalign=True)


@pytest.mark.parametrize("heads,kv_heads,head_dim", [
    (4, 4, 64), (4, 4, 128), (8, 4, 128), (16, 2, 64), (16, 2, 128), (32, 8, 128), (6, 2, 64), (12, 2, 128),
])
def test_packed_groups_and_head_dims(heads, kv_heads, head_dim):
    run(W(f"g{heads // kv_heads}d{head_dim}", (150, 1, 77, 64, 200), heads, kv_heads, head_dim,
          rope_theta=500000.0, seed=2))


@pytest.mark.parametrize("window", [1, 64, 128, 200])
def test_packed_sliding_window(window):
    run(W("window", (260, 90, 333), 64, 8, 64, rope_theta=150000.0, window=window, seed=3))


def test_packed_sinks_gpt_oss_shape():
    sinks = list(np.random.default_rng(4).normal(0.0, 2.0, 64))
    run(W("sinks", (200, 129, 64), 64, 8, 64, rope_theta=150000.0, window=128, seed=4), sinks=sinks)


def test_packed_shuffled_segment_ids():
    run(W("ids", (50, 90, 30, 64, 65), 16, 4, 64, shuffle_ids=True, seed=5))


def test_packed_large_logits_rescale_path():
    run(W("rescale", (1000, 300), 32, 8, 128, rope_theta=500000.0, seed=6), q_scale=16.0)


def test_packed_positions_offset_from_zero():
    def shift(a):
        a["positions"] = a["positions"] + np.int32(37)
        return a
    run(W("offset", (100, 60), 8, 2, 128, seed=7), transform=shift)


def test_packed_tokens_in_any_order():
    # sequences scattered through the pack: the general layout
    def scatter(a):
        perm = np.random.default_rng(8).permutation(len(a["positions"]))
        return {k: np.ascontiguousarray(v[perm]) for k, v in a.items()}
    run(W("scattered", (90, 45, 130), 16, 4, 64, seed=8), transform=scatter)


def test_packed_one_sequence_in_two_runs():
    # the same segment id on two separate runs: tokens attend across both
    def split(a):
        seg = a["segments"].copy()
        seg[150:] = seg[0]             # third sequence takes the first's id
        a["segments"] = seg
        return a
    run(W("two_runs", (100, 50, 80), 8, 2, 64, seed=9), transform=split)


def test_packed_full_size_whole_sequences():
    # the Llama-3.1-8B packed row (8192 tokens); the oracle runs the longest
    # sequence, a middle one and the two shortest alone (a sequence sees only
    # its own tokens), its tokens on all host cores
    w = wl.PACKED_LLAMA
    t = wl.generate_packed(w, "cpu")
    a = {k: wl.to_numpy(v) for k, v in t.items()}
    out = gpu_packed(w, a).cpu()
    shape = oracle.make_shape(0, w.heads, w.kv_heads, w.head_dim, 1, 1, oracle.BF16, rope_theta=w.rope_theta)
    starts = np.concatenate([[0], np.cumsum(w.lengths)])
    order = np.argsort(w.lengths)
    oracle.set_threads(os.cpu_count() or 1)
    try:
        for s in (order[-1], order[len(order) // 2], order[0], order[1]):
            lo, hi = starts[s], starts[s + 1]
            sub = {k: np.ascontiguousarray(v[lo:hi]) for k, v in a.items()}
            _, _, _, o64, rc = oracle.packed(shape, sub["q"], sub["k"], sub["v"], sub["positions"], sub["segments"])
            assert rc == 0
            assert_close(out[lo:hi], o64, "bf16", f"sequence {s} ({hi - lo} tokens)")
    finally:
        oracle.set_threads(1)


def test_packed_attend_reruns_the_attention_bit_for_bit():
    # 66 tiles x 8 kv heads = 528 units: several per CTA from the rewound cursor
    b = binding()
    w = W("again", (3000, 1200), 32, 8, 128, rope_theta=500000.0, seed=10)
    d = to_dev({k: wl.to_numpy(v) for k, v in wl.generate_packed(w, "cpu").items()})
    cos, sin = b.rope_tables(w.rope_theta, w.head_dim, w.max_seq, torch.bfloat16)
    p = b.make_params(1, w.heads, w.kv_heads, w.head_dim, 1, 1, torch.bfloat16, rope_cos=cos, rope_sin=sin)
    ws = b.new_packed_workspace(p, w.tokens)
    out1, out2 = torch.empty_like(d["q"]), torch.full_like(d["q"], float("nan"))
    b.packed(p, d["q"], d["k"], d["v"], d["positions"], d["segments"], out1, ws)
    for _ in range(3):
        out2.fill_(float("nan"))
        b.packed_attend(p, d["v"], d["positions"], out2, ws)
        b.check_status(ws)
        assert b.last_launch_count() == 1
        assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


@pytest.mark.parametrize("scatter,window,head_dim", [(False, 0, 128), (True, 0, 128), (False, 100, 128),
                                                      (True, 100, 128), (False, 0, 64), (True, 100, 64)])
def test_packed_non_finite_keys_and_values_stay_in_their_sequence(scatter, window, head_dim):
    # K and V of one sequence hold inf / NaN: that sequence's outputs are
    # undefined, every other sequence's must match the oracle (its keys never
    # see them: masked scores, zeroed V rows in the shared key blocks)
    w = W("poison", (70, 150, 90, 200), 32, 8, head_dim, rope_theta=500000.0, window=window, seed=11)
    t = wl.generate_packed(w, "cpu")
    a = {k: wl.to_numpy(v) for k, v in t.items()}
    starts = np.concatenate([[0], np.cumsum(w.lengths)])
    bad = np.zeros(len(a["positions"]), dtype=bool)
    bad[starts[1]:starts[2]] = True
    a["k"][bad, :, 1::2] = oracle.f32_to_bf16_bits(float("nan"))
    a["v"][bad, :, ::3] = oracle.f32_to_bf16_bits(float("inf"))
    a["v"][bad, :, 1::3] = oracle.f32_to_bf16_bits(float("nan"))
    if scatter:
        perm = np.random.default_rng(12).permutation(len(bad))
        a = {k: np.ascontiguousarray(v[perm]) for k, v in a.items()}
        bad = bad[perm]
    shape = oracle.make_shape(0, w.heads, w.kv_heads, w.head_dim, 1, 1, oracle.BF16, window=w.window,
                              rope_theta=w.rope_theta)
    _, _, _, out64, rc = oracle.packed(shape, a["q"], a["k"], a["v"], a["positions"], a["segments"])
    assert rc == 0
    out = gpu_packed(w, a).cpu()
    good = np.flatnonzero(~bad)
    assert np.isfinite(out64[good]).all()
    assert_close(out[torch.from_numpy(good)], out64[good], "bf16", "sequences beside the non-finite one")
