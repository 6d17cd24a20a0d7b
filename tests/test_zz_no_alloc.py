"""pdattn_decode_fused_noalloc: the fused step for callers that cannot
allocate device memory, with its scratch in the library's fixed array.

It must give the same result as pdattn_decode_fused with a caller workspace
and as the oracle, call after call (the array keeps the previous call's
contents), including a process's very first call made on a non-blocking
stream, and refuse parameters whose scratch would not fit.  The file is named
so that pytest collects it last.
"""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_step_gb300 import workloads as wl

from gpu_util import binding, gpu_params, oracle_shape, rope_tables_for, assert_close, TOL

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SMALL = wl.Workload("noalloc", rows=6, heads=32, kv_heads=8, head_dim=128, pages_per_row=12, dtype="bf16",
                    rope_theta=500000.0, positions="fixed", fixed_positions=(767, 700, 64, 0, 400, 130), seed=11)


def _case(chunk_pages):
    b = binding()
    w = SMALL
    t = {k: v.cuda() for k, v in wl.generate(w, "cpu").items()}
    tables = rope_tables_for(b, w)
    p = gpu_params(b, w, t["k_pool"].shape[0], tables, chunk_pages=chunk_pages)
    return b, w, t, p


def _noalloc(b, p, t, out, stream=None):
    ptr = lambda x: ctypes.c_void_p(x.data_ptr())
    s = torch.cuda.current_stream() if stream is None else stream
    rc = b.lib.pdattn_decode_fused_noalloc(ctypes.byref(p), ptr(t["q"]), ptr(t["k_new"]), ptr(t["v_new"]),
                                           ptr(t["positions"]), ptr(t["table"]), ptr(t["k_pool"]),
                                           ptr(t["v_pool"]), ptr(out), ctypes.c_void_p(s.cuda_stream))
    assert rc == 0, b.lib.pdattn_last_error()


@pytest.mark.parametrize("chunk_pages", [0, 2])
def test_noalloc_matches_workspace_call_twice_in_a_row(chunk_pages):
    b, w, t, p = _case(chunk_pages)
    ws = b.new_workspace(p)
    ref = torch.empty_like(t["q"])
    b.decode_fused(p, t["q"], t["k_new"], t["v_new"], t["positions"], t["table"], t["k_pool"], t["v_pool"], ref, ws)
    b.check_status(ws)
    mx, mean = TOL[w.dtype]
    for _ in range(2):
        out = torch.full_like(t["q"], float("nan"))
        _noalloc(b, p, t, out)
        torch.cuda.synchronize()
        err = (out.float() - ref.float()).abs()
        assert torch.isfinite(out.float()).all()
        assert err.max().item() <= mx and err.mean().item() <= mean


def test_noalloc_serving_batch_matches_the_oracle_twice_in_a_row():
    # the Llama-3.1-8B serving batch (256 rows, about 10.6 MiB of scratch)
    b = binding()
    w = wl.LLAMA_SERVING
    t = wl.generate(w, "cuda")
    host = {k: wl.to_numpy(v) for k, v in t.items()}
    num_pages = host["k_pool"].shape[0]
    p = gpu_params(b, w, num_pages, rope_tables_for(b, w))
    assert b.workspace_size(p) <= 16 << 20
    kp, vp = host["k_pool"], host["v_pool"]
    oracle.set_threads(os.cpu_count() or 1)
    try:
        _, _, out64, rc = oracle.step(oracle_shape(w, num_pages), host["q"], host["k_new"], host["v_new"],
                                      host["positions"], host["table"], kp, vp)
    finally:
        oracle.set_threads(1)
    assert rc == 0
    for _ in range(2):
        out = torch.full_like(t["q"], float("nan"))
        _noalloc(b, p, t, out)
        torch.cuda.synchronize()
        assert_close(out, out64, w.dtype, "noalloc serving batch")
    assert np.array_equal(wl.to_numpy(t["k_pool"]).view(np.uint8), kp.view(np.uint8))
    assert np.array_equal(wl.to_numpy(t["v_pool"]).view(np.uint8), vp.view(np.uint8))


_FIRST_CALL = r"""
import ctypes, sys
import numpy as np
import torch
sys.path.insert(0, {root!r})
sys.path.insert(0, {tests!r})
import oracle
from paged_gqa_decode_step_gb300 import binding as b
from paged_gqa_decode_step_gb300 import workloads as wl
from gpu_util import gpu_params, oracle_shape, rope_tables_for, assert_close
import test_zz_no_alloc as T

w = T.SMALL
host = {{k: wl.to_numpy(v) for k, v in wl.generate(w, "cpu").items()}}
t = {{k: v.cuda() for k, v in wl.generate(w, "cpu").items()}}
p = gpu_params(b, w, host["k_pool"].shape[0], rope_tables_for(b, w))
torch.cuda.synchronize()
side = torch.cuda.Stream()                      # non-blocking with respect to the legacy stream
out = torch.full_like(t["q"], float("nan"))
with torch.cuda.stream(side):
    T._noalloc(b, p, t, out, stream=side)       # the process's first no-allocation call
side.synchronize()
ws = b.new_workspace(p)
ref = torch.empty_like(t["q"])
b.decode_fused(p, t["q"], t["k_new"], t["v_new"], t["positions"], t["table"], t["k_pool"], t["v_pool"], ref, ws)
b.check_status(ws)
kp, vp = host["k_pool"].copy(), host["v_pool"].copy()
_, _, out64, rc = oracle.step(oracle_shape(w, kp.shape[0]), host["q"], host["k_new"], host["v_new"],
                              host["positions"], host["table"], kp, vp)
assert rc == 0
assert_close(out, out64, w.dtype, "first call on a side stream")
err = (out.float() - ref.float()).abs()
assert err.max().item() <= 2e-2 and err.mean().item() <= 2e-3
print("first-call ok")
"""


def test_noalloc_first_call_of_a_process_on_a_non_blocking_stream():
    binding()    # builds the library if needed
    code = _FIRST_CALL.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "first-call ok" in r.stdout


def test_noalloc_refuses_parameters_that_do_not_fit():
    b, w, t, p = _case(0)
    big = b.make_params(65536, 64, 8, 128, 128, t["k_pool"].shape[0], torch.bfloat16)
    null = ctypes.c_void_p(0)
    dummy = ctypes.c_void_p(t["q"].data_ptr())
    rc = b.lib.pdattn_decode_fused_noalloc(ctypes.byref(big), *([dummy] * 8), null)
    assert rc == b.EINVAL
    assert b"static array" in b.lib.pdattn_last_error()
    assert b.last_launch_count() == 0
