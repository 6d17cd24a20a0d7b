"""Golden fixtures (CPU only).

* ``golden/model_shapes.txt`` holds the attention shapes the model pages
  print; the synthetic workloads must use exactly those.
* ``golden/tiny_step.txt`` is the oracle's own result for the tiny workload,
  written by ``golden/make_tiny_golden.py``; it guards the oracle against
  unintended change.
"""
import os

import numpy as np

from paged_gqa_decode_step_gb300 import workloads as wl

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_shapes():
    shapes = {}
    for line in open(os.path.join(HERE, "model_shapes.txt")):
        line = line.split("--")[0].strip()
        if not line or line.startswith("#"):
            continue
        model, key, value = line.split()
        shapes.setdefault(model, {})[key] = value
    return shapes


def test_workloads_use_the_printed_shapes():
    s = read_shapes()
    ll = s["llama-3.1-8b-instruct"]
    for w in (wl.LLAMA_LAYER, wl.LLAMA_SERVING):
        assert w.heads == int(ll["Heads"]) and w.kv_heads == int(ll["KvHeads"])
        assert w.head_dim == int(ll["H"]) // int(ll["Heads"])
        assert w.max_seq == int(ll["MaxSeq"]) and wl.PAGE_SIZE == int(ll["PageSize"])
        assert w.rope_theta == float(ll["THETA"])
    go = s["gpt-oss-20b"]
    for w in (wl.GPTOSS_FULL, wl.GPTOSS_SLIDING):
        assert (w.heads, w.kv_heads, w.head_dim, w.max_seq) == (
            int(go["Heads"]), int(go["KvHeads"]), int(go["HeadDim"]), int(go["MaxSeq"]))
    assert wl.GPTOSS_SLIDING.window == int(go["Window"]) and wl.GPTOSS_FULL.window == 0
    g2 = s["gpt2"]
    w = wl.GPT2
    assert w.heads == w.kv_heads == int(g2["Heads"])
    assert w.head_dim == int(g2["H"]) // int(g2["Heads"]) and w.max_seq == int(g2["MaxSeq"])
    assert w.dtype == g2["T"] and w.rope_theta <= 0


def read_tiny():
    arrays, name, shape, vals = {}, None, None, []
    for line in open(os.path.join(HERE, "tiny_step.txt")):
        if line.startswith("#"):
            continue
        parts = line.split()
        if parts and not all(len(p) == 4 for p in parts):
            if name:
                arrays[name] = np.array(vals, dtype=np.uint16).reshape(shape)
            name, shape, vals = parts[0], tuple(int(x) for x in parts[1:]), []
        else:
            vals += [int(p, 16) for p in parts]
    arrays[name] = np.array(vals, dtype=np.uint16).reshape(shape)
    return arrays


def test_oracle_reproduces_tiny_golden():
    import importlib.util
    spec = importlib.util.spec_from_file_location("mk", os.path.join(HERE, "make_tiny_golden.py"))
    mk = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mk)
    q_rot, out = mk.compute()
    g = read_tiny()
    assert np.array_equal(g["q_rot"], q_rot)
    assert np.array_equal(g["out"], out)


def test_generator_is_deterministic_and_shaped():
    a = wl.generate(wl.TINY, "cpu")
    b = wl.generate(wl.TINY, "cpu")
    for k in a:
        assert a[k].dtype == b[k].dtype and bool((a[k].view(-1) == b[k].view(-1)).all() | (a[k] != a[k]).any())
    assert a["positions"].tolist() == [37, 100]
    assert a["k_pool"].shape == (16, 8, 64, 64)
    t = a["table"]
    assert (t[0, 1:] == -1).all() and (t[1, 2:] == -1).all()
    used = t[t >= 0].tolist()
    assert len(set(used)) == len(used) == 3
