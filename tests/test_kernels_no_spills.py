"""The decode and tensor-core attention kernels compile for sm_103a without
register spills.

Both hold their working set in registers by design (the decode consumers'
score and output tiles; the tensor-core softmax's 128-key row of S, under a
register hand-over between warpgroups), and a spill there costs far more
than the instructions it saves.  CPU only: nvcc cross-compiles, and the test
reads ptxas's resource report.
"""
import os
import re
import subprocess
import tempfile

import pytest

from paged_gqa_decode_step_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "paged_gqa_decode_step_gb300", "csrc")


@pytest.mark.parametrize("source", ["attend.cu", "prefill.cu"])
def test_kernels_compile_without_spills(source):
    try:
        cc = build.nvcc()
    except RuntimeError:
        pytest.skip("nvcc not found")
    with tempfile.TemporaryDirectory() as d:
        r = subprocess.run([cc, "-c", os.path.join(CSRC, source), "-o", os.path.join(d, "k.o"), "-Xptxas", "-v"]
                           + build._flags(), capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    report = r.stdout + r.stderr
    spills = re.findall(r"(\d+) bytes spill stores, (\d+) bytes spill loads", report)
    assert spills, "no ptxas resource report"
    bad = [s for s in spills if s != ("0", "0")]
    assert not bad, f"{source}: register spills {bad}"
