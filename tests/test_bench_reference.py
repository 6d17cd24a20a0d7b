"""The benchmark's reference arm (the CPU oracle on the host cores) prints one
JSON line with the keys the benchmark contract asks for, and the benchmark
refuses fewer than three warm-up steps.

CPU only: the reference arm times the oracle and launches no kernel.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
REQUIRED = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
            "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e")


def bench(*args):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          timeout=600, cwd=ROOT)


@pytest.mark.parametrize("workload,unit,steps", [
    ("tiny", "GB/s", 2),                 # decode, whole workload per step
    ("llama8b_prefill", "TFLOP/s", 1),   # sampled tokens of the full-size prefill
    ("llama8b_packed", "TFLOP/s", 1),    # the shortest sequences of the full-size pack
])
def test_reference_arm_prints_one_contract_line(workload, unit, steps):
    r = bench("--impl", "reference", "--workload", workload, "--steps", str(steps), "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    for k in REQUIRED:
        assert k in d, k
    assert d["impl"] == "reference" and d["unit"] == unit and d["value"] > 0
    assert d["steps"] == steps and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["higher_is_better"] is True and d["vs_baseline"] is None and d["scaling"] == "weak"
    assert d["config"]["workload"] == workload and d["ms_per_step"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == unit
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_fewer_than_three_warmup_steps_are_refused():
    r = bench("--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "2")
    assert r.returncode != 0
    assert "warmup" in r.stderr


def test_our_arm_fails_loudly_without_a_gpu():
    # no CPU fallback: without a CUDA device the timed arm exits with an error
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    r = bench("--steps", "3", "--warmup", "3")
    assert r.returncode != 0
    assert not [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
