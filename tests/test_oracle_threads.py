"""The oracle's rows may run on several threads (OpenMP): the results must be
those of the serial loop, bit for bit, including the reported status."""
import numpy as np

import oracle
from paged_gqa_decode_step_gb300 import workloads as wl


def test_rows_on_threads_match_the_serial_loop():
    w = wl.Workload("threads", rows=24, heads=8, kv_heads=2, head_dim=64, pages_per_row=6, dtype="bf16",
                    positions="uniform", pos_lo=0, pos_hi=383, window=0, rope_theta=10000.0, seed=41)
    t = wl.generate(w, "cpu")
    a = {k: wl.to_numpy(v) for k, v in t.items()}
    shape = oracle.make_shape(w.rows, w.heads, w.kv_heads, w.head_dim, w.pages_per_row, a["k_pool"].shape[0],
                              oracle.BF16, rope_theta=w.rope_theta)
    a["table"][5, :] = -1            # a bad row: its status must still be reported
    runs = []
    try:
        for n in (1, 4):
            oracle.set_threads(n)
            kp, vp = a["k_pool"].copy(), a["v_pool"].copy()
            runs.append(oracle.step(shape, a["q"], a["k_new"], a["v_new"], a["positions"], a["table"], kp, vp))
    finally:
        oracle.set_threads(1)
    (q1, o1, d1, rc1), (q4, o4, d4, rc4) = runs
    assert rc1 == rc4 != 0
    assert np.array_equal(q1, q4) and np.array_equal(o1, o4)
    assert np.array_equal(d1.view(np.uint64), d4.view(np.uint64))


def test_packed_tokens_on_threads_match_the_serial_loop():
    w = wl.PackedWorkload("threads", lengths=(70, 33, 90), heads=8, kv_heads=2, head_dim=64, window=40,
                          shuffle_ids=True, seed=42)
    a = {k: wl.to_numpy(v) for k, v in wl.generate_packed(w, "cpu").items()}
    shape = oracle.make_shape(0, w.heads, w.kv_heads, w.head_dim, 1, 1, oracle.BF16, window=w.window,
                              rope_theta=w.rope_theta)
    runs = []
    try:
        for n in (1, 4):
            oracle.set_threads(n)
            runs.append(oracle.packed(shape, a["q"], a["k"], a["v"], a["positions"], a["segments"]))
    finally:
        oracle.set_threads(1)
    (q1, k1, o1, d1, rc1), (q4, k4, o4, d4, rc4) = runs
    assert rc1 == rc4 == 0
    assert np.array_equal(q1, q4) and np.array_equal(k1, k4) and np.array_equal(o1, o4)
    assert np.array_equal(d1.view(np.uint64), d4.view(np.uint64))
