"""pdattn_decode_fused_noalloc: the fused step for callers that cannot
allocate device memory, with its scratch in the library's fixed array.

It must give the same result as pdattn_decode_fused with a caller workspace,
call after call (the array keeps the previous call's contents), and refuse
parameters whose scratch would not fit.  The file is named so that pytest
collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from paged_gqa_decode_step_gb300 import workloads as wl

from gpu_util import binding, gpu_params, rope_tables_for, TOL

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


def _case(chunk_pages):
    b = binding()
    w = wl.Workload("noalloc", rows=6, heads=32, kv_heads=8, head_dim=128, pages_per_row=12, dtype="bf16",
                    rope_theta=500000.0, positions="fixed", fixed_positions=(767, 700, 64, 0, 400, 130), seed=11)
    t = {k: v.cuda() for k, v in wl.generate(w, "cpu").items()}
    tables = rope_tables_for(b, w)
    p = gpu_params(b, w, t["k_pool"].shape[0], tables, chunk_pages=chunk_pages)
    return b, w, t, p


def _noalloc(b, p, t, out):
    ptr = lambda x: ctypes.c_void_p(x.data_ptr())
    rc = b.lib.pdattn_decode_fused_noalloc(ctypes.byref(p), ptr(t["q"]), ptr(t["k_new"]), ptr(t["v_new"]),
                                           ptr(t["positions"]), ptr(t["table"]), ptr(t["k_pool"]),
                                           ptr(t["v_pool"]), ptr(out),
                                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
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


def test_noalloc_refuses_parameters_that_do_not_fit():
    b, w, t, p = _case(0)
    big = b.make_params(65536, 64, 8, 128, 128, t["k_pool"].shape[0], torch.bfloat16)
    null = ctypes.c_void_p(0)
    dummy = ctypes.c_void_p(t["q"].data_ptr())
    rc = b.lib.pdattn_decode_fused_noalloc(ctypes.byref(big), *([dummy] * 8), null)
    assert rc == b.EINVAL
    assert b"static array" in b.lib.pdattn_last_error()
    assert b.last_launch_count() == 0
