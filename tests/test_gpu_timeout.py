"""A bounded device wait that runs out, provoked without any fault.

Every mbarrier wait of the decode attention kernel gives up after about two
seconds, records PDATTN_ETIMEOUT in the workspace's status word and lets the
kernel wind down (its copies in flight land first).  The control block holds
a test hook that calls never set: with it, CTA 0 leaves the first stage of
its first item unissued, so its consumers wait on a barrier that nothing
completes.  The test checks that the status reports the timeout, that the
context stays usable, that the withdrawn plan is refused for attention-only
calls, and that the next planned call (and a call on a fresh workspace) is
oracle-exact again.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_step_gb300 import workloads as wl

from gpu_util import binding, gpu_params, oracle_shape, rope_tables_for, assert_close

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]

# Byte offset of the control block's test hook (the int after the plan header:
# status, cursor, done count, items, chunk pages, magic, rows, kv heads, pages
# per row, max items, group, head dim, grid).
CTRL_TEST_HOLD = 13 * 4


def _set_hold(ws, value):
    ws[CTRL_TEST_HOLD:CTRL_TEST_HOLD + 4].view(torch.int32).fill_(value)


def _case():
    w = wl.Workload("timeout", rows=24, heads=32, kv_heads=8, head_dim=128, pages_per_row=16, dtype="bf16",
                    rope_theta=500000.0, positions="uniform", pos_lo=100, pos_hi=1023, seed=77)
    t = wl.generate(w, "cpu")
    host = {k: wl.to_numpy(v) for k, v in t.items()}
    num_pages = host["k_pool"].shape[0]
    kp, vp = host["k_pool"].copy(), host["v_pool"].copy()
    _, _, out64, rc = oracle.step(oracle_shape(w, num_pages), host["q"], host["k_new"], host["v_new"],
                                  host["positions"], host["table"], kp, vp)
    assert rc == 0
    return w, {k: v.cuda() for k, v in t.items()}, num_pages, out64


def test_a_wait_that_runs_out_is_reported_and_the_context_stays_usable():
    b = binding()
    w, d, num_pages, out64 = _case()
    p = gpu_params(b, w, num_pages, rope_tables_for(b, w))
    ws = b.new_workspace(p)
    q_rot = torch.empty_like(d["q"])
    out = torch.zeros_like(d["q"])
    b.rope_write_kv(p, d["q"], d["k_new"], d["v_new"], d["positions"], d["table"], q_rot, d["k_pool"],
                    d["v_pool"], ws)
    b.plan(p, d["positions"], ws)
    _set_hold(ws, 1)
    b.attend(p, q_rot, d["positions"], d["table"], d["k_pool"], d["v_pool"], out, ws)
    with pytest.raises(b.PdattnError) as e:
        b.check_status(ws)
    assert e.value.status == b.ETIMEOUT

    # the plan was withdrawn: attention alone on it is refused on the device
    _set_hold(ws, 0)
    b.attend(p, q_rot, d["positions"], d["table"], d["k_pool"], d["v_pool"], out, ws)
    with pytest.raises(b.PdattnError) as e:
        b.check_status(ws)
    assert e.value.status == b.EINVAL

    # planning again makes the same workspace usable
    out.fill_(float("nan"))
    b.plan(p, d["positions"], ws)
    b.attend(p, q_rot, d["positions"], d["table"], d["k_pool"], d["v_pool"], out, ws)
    b.check_status(ws)
    assert_close(out, out64, w.dtype, "after re-planning")

    # and a fused step on a fresh workspace is exact
    ws2 = b.new_workspace(p)
    out.fill_(float("nan"))
    b.decode_fused(p, d["q"], d["k_new"], d["v_new"], d["positions"], d["table"], d["k_pool"], d["v_pool"],
                   out, ws2)
    b.check_status(ws2)
    assert_close(out, out64, w.dtype, "fresh workspace")


def test_the_fused_step_reports_a_timeout_and_recovers_on_the_next_call():
    b = binding()
    w, d, num_pages, out64 = _case()
    p = gpu_params(b, w, num_pages, rope_tables_for(b, w))
    ws = b.new_workspace(p)
    out = torch.zeros_like(d["q"])
    _set_hold(ws, 1)
    b.decode_fused(p, d["q"], d["k_new"], d["v_new"], d["positions"], d["table"], d["k_pool"], d["v_pool"],
                   out, ws)
    with pytest.raises(b.PdattnError) as e:
        b.check_status(ws)
    assert e.value.status == b.ETIMEOUT
    _set_hold(ws, 0)
    out.fill_(float("nan"))
    b.decode_fused(p, d["q"], d["k_new"], d["v_new"], d["positions"], d["table"], d["k_pool"], d["v_pool"],
                   out, ws)
    b.check_status(ws)
    assert_close(out, out64, w.dtype, "next call on the same workspace")
    assert np.isfinite(wl.to_numpy(out.float())).all()
