#!/usr/bin/env python
"""Benchmark of one paged GQA decode step (RoPE + cache write + attention).

Default workload: the Llama-3.1-8B serving batch (256 rows, 32 query heads,
8 kv heads, head dim 128, 64-token pages, context lengths log-uniform in
[16, 8192], bf16).  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

* value: KV GB/s of the whole step over all ranks (algorithmic K/V bytes the
  step must read, divided by the device time of K steps; max over ranks).
* roofline: the attention kernel timed alone with CUDA events around each
  launch; achieved = its algorithmic bytes per launch / mean launch time,
  against the measured HBM copy bandwidth.
* e2e: the same metric through the public call with pinned host buffers:
  each step copies that step's inputs host->device and its output back; as
  in a serving loop the next step's copy overlaps the current step
  (double-buffered, copy stream) and the host waits for each output.
* cpu_baseline: the CPU oracle on the host (single thread), timed on whole
  steps of the same workload.
* --impl reference: the CPU oracle alone, each step a bounded sample of rows.

--workload llama8b_prefill measures the paged prefill instead (8 rows x 1024
new tokens on cached prefixes 0 .. 7168, Llama-3.1-8B attention shape): value
= attention TFLOP/s of whole prefill calls (4 * D * heads * visible keys per
token), roofline against the measured bf16 tensor peak.  --workload
llama8b_packed measures packed sequences the same way (one 8192-token row of
eight sequences, no cache).
"""
import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from paged_gqa_decode_step_gb300 import workloads as wl  # noqa: E402

METRIC = "paged decode attention KV GB/s (% of GB300 HBM peak) and row-steps/s per layer"
L2_BYTES = 129 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ helpers --
def visible(w, pos):
    lo = max(0, pos - w.window + 1) if w.window > 0 else 0
    return lo, pos - lo + 1


def kv_bytes(w, positions):
    """K and V bytes the step must read: sum_r 2 * ctx_r * Hk * D * E."""
    return sum(2 * visible(w, int(p))[1] * w.kv_heads * w.head_dim * w.elem_bytes for p in positions)


def attend_bytes(w, positions):
    """Algorithmic bytes of the attention kernel: K/V, q in, out, table entries."""
    E = w.elem_bytes
    total = kv_bytes(w, positions)
    for p in positions:
        lo, _ = visible(w, int(p))
        total += 2 * w.heads * w.head_dim * E + 4 * (int(p) // 64 - lo // 64 + 1)
    return total


def step_bytes(w, positions):
    """Whole step: attention plus q read / rotated q write, k and v in, slot writes."""
    E = w.elem_bytes
    R = len(positions)
    return attend_bytes(w, positions) + R * (2 * w.heads * w.head_dim * E + 4 * w.kv_heads * w.head_dim * E + 8)


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    """Hash of the sources that define the decode attention kernel."""
    h = hashlib.sha256()
    for name in ("attend.cu", "common.cuh", "internal.h"):
        with open(os.path.join(ROOT, "paged_gqa_decode_step_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM bytes per attention launch from the committed ncu summary, if it
    was taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"attend_{workload}_traffic.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("source_hash") != kernel_source_hash():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the GPU works.
    summary() covers every sample; window(t0, t1) only those taken between
    two time.time() stamps (a timed region)."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device):
        self.proc = None
        self.rows = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        sel = []
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            sel = []
        self.cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"] + sel

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def _load(self):
        if self.rows is not None:
            return self.rows
        import datetime
        self.out.flush()
        rows = []
        with open(self.out.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) != 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
                except ValueError:
                    continue
        os.unlink(self.out.name)
        self.rows = rows
        return rows

    def _summarise(self, rows, extra=None):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        reasons = sorted({self.REASONS[i] for _, _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        sm = sorted(r[1] for r in rows)
        d = {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(r[2] for r in rows), "reasons": reasons,
             "samples": len(rows)}
        if extra:
            d.update(extra)
        return d

    def summary(self):
        return self._summarise(self._load())

    def window(self, t0, t1):
        rows = self._load()
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        if inside:
            return self._summarise(inside, {"within_timed_region": True})
        return self._summarise(rows, {"within_timed_region": False})


# ------------------------------------------------------------- end to end --
def e2e_pipelined(dev_tensors, names, run, out, n_steps, world):
    """End-to-end seconds per step through the public call.  Every step copies
    its own inputs (`names`) from pinned host memory and reads its output back
    into pinned host memory.  As in a serving loop, inputs and outputs are
    double-buffered, the copies run on their own streams (host to device
    ahead of the step, device to host after it) under the neighbouring steps'
    compute, and the host waits for step i - 1's output while step i runs.
    `run(inputs, out)` issues the library call on the current stream.
    Returns (seconds per step, H2D bytes per step, D2H bytes per step)."""
    host = [{k: dev_tensors[k].cpu().pin_memory() for k in names} for _ in range(2)]
    dev = [{k: torch.empty_like(dev_tensors[k]) for k in names} for _ in range(2)]
    outs = [torch.empty_like(out) for _ in range(2)]
    host_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
    compute = torch.cuda.current_stream()
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    inputs_free = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    out_ready = [torch.cuda.Event() for _ in range(2)]
    for e in inputs_free + out_ready:
        e.record(compute)

    def h2d(i):
        b = i % 2
        h2d_stream.wait_event(inputs_free[b])           # the step two back is done with this buffer
        with torch.cuda.stream(h2d_stream):
            for k in names:
                dev[b][k].copy_(host[b][k], non_blocking=True)
        h2d_done[b].record(h2d_stream)

    def step(i):
        b = i % 2
        compute.wait_event(h2d_done[b])
        compute.wait_event(out_ready[b])                # the step two back has read its output out
        run(dev[b], outs[b])
        inputs_free[b].record(compute)
        computed[b].record(compute)
        d2h_stream.wait_event(computed[b])
        with torch.cuda.stream(d2h_stream):
            host_out[b].copy_(outs[b], non_blocking=True)
        out_ready[b].record(d2h_stream)

    def loop(n):
        torch.cuda.synchronize()
        barrier(world)
        t0 = time.perf_counter()
        h2d(0)
        for i in range(n):
            if i + 1 < n:
                h2d(i + 1)
            step(i)
            if i >= 1:
                out_ready[(i - 1) % 2].synchronize()    # step i - 1's output is on the host
        out_ready[(n - 1) % 2].synchronize()
        return time.perf_counter() - t0

    loop(3)
    secs = loop(n_steps) / n_steps
    h2d_bytes = sum(v.numel() * v.element_size() for v in host[0].values())
    return secs, h2d_bytes, host_out[0].numel() * host_out[0].element_size()


# ------------------------------------------------------------- timing --
def device_ms(fn, n, flush=None):
    """Mean device milliseconds of n calls of fn on the current stream.  Without
    `flush` (inputs larger than L2) one pair of CUDA events brackets all n
    calls; with it, a pair brackets each call and L2 is flushed (a write of
    `flush`, outside the events) before each."""
    torch.cuda.synchronize()
    if flush is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for e0, e1 in evs:
        flush.fill_(1)
        e0.record()
        fn()
        e1.record()
    torch.cuda.synchronize()
    return sum(e0.elapsed_time(e1) for e0, e1 in evs) / n


def keep_busy(fn, seconds, flush=None):
    """Untimed calls of fn for about `seconds` of wall time, so that the clock
    samples around a short timed region see the GPU under this load."""
    t_end = time.time() + seconds
    i = 0
    while time.time() < t_end:
        if flush is not None:
            flush.fill_(1)
        fn()
        i += 1
        if i % 32 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()


# -------------------------------------------------------------- distributed --
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def rank_seed(w, rank):
    """Each rank draws its own batch of rows (weak scaling, no data exchange)."""
    return w.seed + 7919 * rank


# --------------------------------------------------------------------- CPU --
def cpu_oracle_rate(w, host, budget_s, rows_per_step=None, max_steps=None, threads=1):
    """Run the oracle on whole steps (or row samples) for about budget_s, its
    rows on `threads` threads.  Returns (KV GB/s, seconds, description, steps)."""
    import numpy as np
    import oracle
    threads = oracle.set_threads(threads)
    pos = host["positions"]
    R = len(pos)
    num_pages = host["k_pool"].shape[0]
    od = oracle.BF16 if w.dtype == "bf16" else oracle.F32
    done_bytes, spent, steps, start_row = 0, 0.0, 0, 0
    rows_per_step = rows_per_step or R
    while True:
        sub = (np.arange(rows_per_step) + start_row) % R
        start_row = (start_row + rows_per_step) % R
        shape = oracle.make_shape(len(sub), w.heads, w.kv_heads, w.head_dim, w.pages_per_row, num_pages, od,
                                  window=w.window, rope_theta=w.rope_theta)
        args = [np.ascontiguousarray(host[k][sub]) for k in ("q", "k_new", "v_new", "positions", "table")]
        t0 = time.perf_counter()
        _, _, _, rc = oracle.step(shape, *args, host["k_pool"], host["v_pool"])
        spent += time.perf_counter() - t0
        assert rc == 0
        done_bytes += kv_bytes(w, pos[sub])
        steps += 1
        if (max_steps and steps >= max_steps) or (not max_steps and spent >= budget_s):
            break
    desc = (f"{steps} oracle step(s) of {rows_per_step} of the {R} rows "
            f"({'whole workload' if rows_per_step == R else 'rows taken round-robin'}), "
            f"{'single thread' if threads == 1 else f'rows on {threads} threads'}")
    oracle.set_threads(1)
    return done_bytes / spent / 1e9, spent, desc, steps


# --------------------------------------------------- the other configs --
DECODE_EXTRAS = ("llama8b_layer", "gptoss20b_full", "gptoss20b_sliding", "gpt2_f32")


def measure_decode_config(args, b, w, dev, world, rank):
    """One decode workload in light form: whole fused steps (CUDA events, L2
    flushed unless the K/V outgrows it), the attention kernel alone against
    the HBM roofline, and the clocks seen while the steps ran."""
    t = wl.generate(w, dev, seed=rank_seed(w, rank))
    pos_list = t["positions"].cpu().tolist()
    num_pages = t["k_pool"].shape[0]
    tables = b.rope_tables(w.rope_theta, w.head_dim, w.max_seq, w.torch_dtype) if w.rope_theta > 0 else (None, None)
    p = b.make_params(w.rows, w.heads, w.kv_heads, w.head_dim, w.pages_per_row, num_pages, w.torch_dtype,
                      window=w.window, rope_cos=tables[0], rope_sin=tables[1])
    ws = b.new_workspace(p)
    out = torch.empty_like(t["q"])
    kvb = kv_bytes(w, pos_list)
    large = kvb > 2 * L2_BYTES
    flush = None if large else torch.empty(4 * L2_BYTES // 4, dtype=torch.int32, device=dev)

    def step():
        b.decode_fused(p, t["q"], t["k_new"], t["v_new"], t["positions"], t["table"], t["k_pool"], t["v_pool"], out, ws)

    for _ in range(args.warmup):
        step()
    b.check_status(ws)
    with ClockSampler(dev) as clocks:
        t_load = time.time()
        if not args.quick:
            keep_busy(step, 0.3, flush)
        barrier(world)
        ms = device_ms(step, args.steps, flush)
        t_end = time.time()
        barrier(world)
    clk = clocks.window(t_load, t_end)
    b.check_status(ws)
    ms = max_over_ranks(ms, world)
    all_kv = sum_over_ranks(kvb, world)

    q_rot = torch.empty_like(t["q"])
    b.rope_write_kv(p, t["q"], t["k_new"], t["v_new"], t["positions"], t["table"], q_rot, t["k_pool"], t["v_pool"], ws)
    b.plan(p, t["positions"], ws)
    att_ms = device_ms(lambda: b.attend(p, q_rot, t["positions"], t["table"], t["k_pool"], t["v_pool"], out, ws),
                       max(20, min(args.steps, 400)), flush)
    b.check_status(ws)
    att_bytes = attend_bytes(w, pos_list)
    peak, peak_kind = measured_hbm_peak()
    achieved = att_bytes / (att_ms * 1e-3) / 1e9
    value = all_kv / (ms * 1e-3) / 1e9
    return {
        "metric": "KV GB/s", "value": value, "unit": "GB/s", "ms_per_step": ms, "steps": args.steps,
        "dtype": w.dtype, "rows": w.rows, "heads": w.heads, "kv_heads": w.kv_heads, "head_dim": w.head_dim,
        "window": w.window, "positions": f"{w.positions} [{w.pos_lo}, {w.pos_hi}]",
        "kv_bytes_per_step": kvb, "row_steps_per_s": w.rows * world / (ms * 1e-3),
        "frac_of_hbm_peak": value / world / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "kernel": f"attend_kernel<{w.dtype},{w.head_dim}>", "bytes_per_launch": att_bytes,
                     "launch_us": att_ms * 1e3, "peak_kind": peak_kind},
        "l2": "inputs larger than L2" if large else "L2 flushed (512 MB write) between timed steps, outside the events",
        "clocks": clk,
    }


def measure_layers(args, b, w, n_layers, dev, world, rank, pairs=True):
    """Decode step over n_layers layers (shared positions and page table,
    per-layer caches): one pdattn_decode_layers call against one decode_fused
    call per layer, back to back on the stream, and against those calls
    replayed from a CUDA graph.  With `pairs` the layers alternate a window-128
    layer and a full one (gpt-oss-20b LayerPairs); otherwise all are full.
    K/V bytes are all layers' visible pages."""
    base = wl.generate(w, dev, seed=rank_seed(w, rank))
    gen = torch.Generator(device=dev)
    gen.manual_seed(rank_seed(w, rank) + 1)
    pos_list = base["positions"].cpu().tolist()
    num_pages = base["k_pool"].shape[0]
    cos, sin = b.rope_tables(w.rope_theta, w.head_dim, w.max_seq, w.torch_dtype)
    windows = [128 if (pairs and l % 2 == 0) else 0 for l in range(n_layers)]
    layers = []
    for l in range(n_layers):
        y = {k: torch.randn(base[k].shape, generator=gen, device=dev, dtype=torch.float32).to(w.torch_dtype)
             for k in ("q", "k_new", "v_new", "k_pool", "v_pool")}
        y["out"] = torch.empty_like(y["q"])
        y["window"] = windows[l]
        layers.append(y)
    p = b.make_params(w.rows, w.heads, w.kv_heads, w.head_dim, w.pages_per_row, num_pages, w.torch_dtype,
                      rope_cos=cos, rope_sin=sin)
    per_layer = [b.make_params(w.rows, w.heads, w.kv_heads, w.head_dim, w.pages_per_row, num_pages, w.torch_dtype,
                               window=windows[l], rope_cos=cos, rope_sin=sin) for l in range(n_layers)]
    ws = b.new_layers_workspace(p, n_layers)
    ws_l = [b.new_workspace(q) for q in per_layer]
    kvb = sum(kv_bytes(replace_window(w, windows[l]), pos_list) for l in range(n_layers))
    large = kvb > 2 * L2_BYTES
    flush = None if large else torch.empty(4 * L2_BYTES // 4, dtype=torch.int32, device=dev)

    def fused():
        b.decode_layers(p, layers, base["positions"], base["table"], ws)

    def separate():
        for l, y in enumerate(layers):
            b.decode_fused(per_layer[l], y["q"], y["k_new"], y["v_new"], base["positions"], base["table"],
                           y["k_pool"], y["v_pool"], y["out"], ws_l[l])

    res = {}
    for name, fn in (("one_call", fused), ("per_layer_calls", separate)):
        for _ in range(args.warmup):
            fn()
        with ClockSampler(dev) as clocks:
            t_load = time.time()
            keep_busy(fn, 0.3, flush)
            ms = device_ms(fn, args.steps, flush)
            t_end = time.time()
        res[name] = {"ms_per_step": ms, "kv_gbs": kvb / (ms * 1e-3) / 1e9, "clocks": clocks.window(t_load, t_end)}
    b.check_status(ws)
    for q in ws_l:
        b.check_status(q)
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            separate()
        for _ in range(3):
            graph.replay()
        ms = device_ms(graph.replay, args.steps, flush)
        res["per_layer_calls_graph"] = {"ms_per_step": ms, "kv_gbs": kvb / (ms * 1e-3) / 1e9}
        del graph
    except Exception as exc:  # an extra measurement; the two above stand on their own
        print(f"graph capture skipped: {exc}", file=sys.stderr)
    peak, peak_kind = measured_hbm_peak()
    return {"layers": n_layers, "windows": "128, 0, 128, 0, ..." if pairs else "0 (all full)", "rows": w.rows,
            "heads": w.heads,
            "kv_heads": w.kv_heads, "head_dim": w.head_dim, "kv_bytes_per_step": kvb,
            "frac_of_hbm_peak": res["one_call"]["kv_gbs"] / peak, "peak": peak, "peak_kind": peak_kind,
            "l2": "inputs larger than L2" if large else "L2 flushed (512 MB write) between timed steps",
            **res}


def replace_window(w, window):
    from dataclasses import replace
    return replace(w, window=window)


def other_configs(args, world, rank, local):
    """Every other workload of the step, measured in this process; keyed by name."""
    from paged_gqa_decode_step_gb300 import binding as b
    dev = torch.device("cuda", local)
    res = {}
    for name in DECODE_EXTRAS:
        if name == args.workload:
            continue
        res[name] = measure_decode_config(args, b, wl.WORKLOADS[name], dev, world, rank)
        torch.cuda.empty_cache()
    for n_layers in (2, 24):
        res[f"gptoss20b_layers{n_layers}"] = measure_layers(args, b, wl.GPTOSS_FULL, n_layers, dev, world, rank)
        torch.cuda.empty_cache()
    res["llama8b_layer_layers32"] = measure_layers(args, b, wl.LLAMA_LAYER, 32, dev, world, rank, pairs=False)
    torch.cuda.empty_cache()
    for w in wl.PREFILL_WORKLOADS.values():
        res[w.name] = run_prefill(args, w, world, rank, local, light=True)
        torch.cuda.empty_cache()
    for w in wl.PACKED_WORKLOADS.values():
        res[w.name] = run_packed(args, w, world, rank, local, light=True)
        torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------- our arm --
def run_ours(args, w, world, rank, local):
    from paged_gqa_decode_step_gb300 import build
    build.build()
    from paged_gqa_decode_step_gb300 import binding as b

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    t = wl.generate(w, dev, seed=rank_seed(w, rank))
    pos_list = t["positions"].cpu().tolist()
    num_pages = t["k_pool"].shape[0]
    tables = b.rope_tables(w.rope_theta, w.head_dim, w.max_seq, w.torch_dtype) if w.rope_theta > 0 else (None, None)
    p = b.make_params(w.rows, w.heads, w.kv_heads, w.head_dim, w.pages_per_row, num_pages, w.torch_dtype,
                      window=w.window, rope_cos=tables[0], rope_sin=tables[1], chunk_pages=args.chunk_pages)
    ws = b.new_workspace(p)
    out = torch.empty_like(t["q"])
    kvb = kv_bytes(w, pos_list)
    pool_bytes = 2 * t["k_pool"].numel() * t["k_pool"].element_size()
    large = kvb > 2 * L2_BYTES
    flush = None if large else torch.empty(4 * L2_BYTES // 4, dtype=torch.int32, device=dev)

    def step():
        b.decode_fused(p, t["q"], t["k_new"], t["v_new"], t["positions"], t["table"], t["k_pool"], t["v_pool"], out, ws)

    for _ in range(args.warmup):
        step()
    b.check_status(ws)
    launches_per_step = b.last_launch_count()

    # ---- timed region: K whole steps (clock samples over a loaded lead-in and the region)
    with ClockSampler(dev) as clocks:
        t_load = time.time()
        if not args.quick:
            keep_busy(step, 0.3, flush)
        barrier(world)
        ms = device_ms(step, args.steps, flush)
        t_end = time.time()
        barrier(world)
    clk = clocks.window(t_load, t_end)
    b.check_status(ws)
    if args.quick:
        # profiling mode: warm-up and timed steps only
        if rank == 0:
            print(json.dumps({"quick": True, "workload": w.name, "chunk_pages": args.chunk_pages,
                              "ms_per_step": ms, "kv_gbs": kvb / (ms * 1e-3) / 1e9}), flush=True)
        return None
    ms = max_over_ranks(ms, world)
    all_kv = sum_over_ranks(kvb, world)
    rows_all = w.rows * world
    value = all_kv / (ms * 1e-3) / 1e9

    # ---- the same step captured once in a CUDA graph and replayed
    graph_ms = None
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_g = max(10, min(args.steps, 1000))
        if large:
            g0.record()
            for _ in range(n_g):
                graph.replay()
            g1.record()
            torch.cuda.synchronize()
            graph_ms = g0.elapsed_time(g1) / n_g
        b.check_status(ws)
        del graph
    except Exception as exc:  # capture is an extra measurement; the step above stands on its own
        print(f"graph capture skipped: {exc}", file=sys.stderr)
    graph_ms = max_over_ranks(graph_ms, world) if graph_ms is not None else None

    # ---- roofline: the attention kernel alone, events around every launch
    q_rot = torch.empty_like(t["q"])
    b.rope_write_kv(p, t["q"], t["k_new"], t["v_new"], t["positions"], t["table"], q_rot, t["k_pool"], t["v_pool"], ws)
    b.plan(p, t["positions"], ws)
    for _ in range(3):
        b.attend(p, q_rot, t["positions"], t["table"], t["k_pool"], t["v_pool"], out, ws)
    att_ms = device_ms(lambda: b.attend(p, q_rot, t["positions"], t["table"], t["k_pool"], t["v_pool"], out, ws),
                       max(20, min(args.steps, 400)), flush)
    b.check_status(ws)
    att_bytes = attend_bytes(w, pos_list)
    peak, peak_kind = measured_hbm_peak()
    achieved = att_bytes / (att_ms * 1e-3) / 1e9
    traffic = profiled_traffic(w.name)

    # ---- end to end: pinned host inputs in, output back, every step
    n_e2e = max(10, min(args.steps, 500))
    e2e_s, h2d, d2h = e2e_pipelined(
        t, ("q", "k_new", "v_new", "positions", "table"),
        lambda d, o: b.decode_fused(p, d["q"], d["k_new"], d["v_new"], d["positions"], d["table"], t["k_pool"],
                                    t["v_pool"], o, ws), out, n_e2e, world)
    e2e_s = max_over_ranks(e2e_s, world)
    b.check_status(ws)
    e2e_value = all_kv / e2e_s / 1e9

    # ---- CPU baseline: the oracle on this host, rank 0 at N = 1 only: one
    # thread, and its rows spread over every core
    cpu = cpu_par = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host = {k: wl.to_numpy(v) for k, v in t.items()}
        rate, spent, desc, _ = cpu_oracle_rate(w, host, args.cpu_baseline_seconds)
        cpu = {"value": rate, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": desc,
               "seconds": round(spent, 2), "cpu": cpu_model()}
        n_cores = os.cpu_count() or 1
        rate, spent, desc, _ = cpu_oracle_rate(w, host, args.cpu_baseline_seconds, threads=n_cores)
        cpu_par = {"value": rate, "unit": "GB/s", "cores": n_cores, "kind": "oracle", "sample": desc,
                   "seconds": round(spent, 2), "cpu": cpu_model()}

    extras = None if args.no_extra else other_configs(args, world, rank, local)

    if rank != 0:
        return None
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic (seeded N(0,1) q/k/v and prefilled pool, shuffled page table)",
        "config": {
            "workload": w.name, "rows_per_gpu": w.rows, "heads": w.heads, "kv_heads": w.kv_heads,
            "head_dim": w.head_dim, "page_size": 64, "pages_per_row": w.pages_per_row,
            "positions": f"{w.positions} [{w.pos_lo}, {w.pos_hi}]", "window": w.window,
            "rope_theta": w.rope_theta, "kv_bytes_per_step_per_gpu": kvb,
            "l2": (f"inputs larger than L2: each step streams {kvb / 1e9:.2f} GB of K/V from a "
                   f"{pool_bytes / 1e9:.2f} GB pool (L2 129 MB)") if large else
                  "L2 flushed (512 MB write) between timed steps, outside the events",
            "parallelism": f"replicas x{world} (rows sharded across ranks, no exchange)",
        },
        "row_steps_per_s": rows_all / (ms * 1e-3),
        "frac_of_hbm_peak": value / world / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "kernel": f"attend_kernel<{w.dtype},{w.head_dim}>",
                     "bytes_per_launch": att_bytes, "launch_us": att_ms * 1e3, "peak_kind": peak_kind},
        "cpu_baseline": cpu,
        "cpu_parallel": cpu_par,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_s * 1e3},
        "graph": None if graph_ms is None else {
            "ms_per_step": graph_ms, "value": all_kv / (graph_ms * 1e-3) / 1e9, "unit": "GB/s",
            "what": "the same step captured once in a CUDA graph and replayed"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "workloads": extras,
    }
    return line


def cpu_model():
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return os.uname().machine


# ----------------------------------------------------------- reference arm --
def run_reference(args, w, world, rank):
    """The oracle on the host cores, each step a bounded sample of rows."""
    if rank != 0:
        return None
    t = wl.generate(w, "cpu", seed=rank_seed(w, 0)) if w.rows * w.pages_per_row <= 4096 else None
    if t is None:
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = wl.generate(w, dev, seed=rank_seed(w, 0))
    host = {k: wl.to_numpy(v) for k, v in t.items()}
    del t
    pos = host["positions"]
    mean_ctx = float(sum(visible(w, int(p))[1] for p in pos)) / len(pos)
    # ~11 us per visible token-row on one core; size each step to fit ~90 s total
    n_cores = os.cpu_count() or 1
    per_step_budget = min(5.0, 90.0 / max(1, args.steps + args.warmup))
    per_row = mean_ctx * w.heads / 32 * 11e-6 * (w.head_dim / 128) / n_cores
    rows = int(max(1, min(w.rows, per_step_budget / max(per_row, 1e-9))))
    if args.warmup:
        cpu_oracle_rate(w, host, 0, rows_per_step=rows, max_steps=args.warmup, threads=n_cores)
    rate, spent, desc, steps = cpu_oracle_rate(w, host, 0, rows_per_step=rows, max_steps=max(1, args.steps),
                                               threads=n_cores)
    ms = spent / steps * 1e3
    return {
        "metric": METRIC, "value": rate, "unit": "GB/s", "n_gpus": world, "steps": steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic", "impl": "reference",
        "config": {"workload": w.name, "rows_per_step": rows, "rows": w.rows},
        "cpu_baseline": {"kind": "oracle", "cores": n_cores, "sample": desc, "value": rate, "unit": "GB/s",
                         "cpu": cpu_model()},
        "e2e": {"value": rate, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------- prefill --
PREFILL_METRIC = "paged prefill attention TFLOP/s (% of GB300 bf16 tensor peak)"


def prefill_flops(w, positions):
    """4 * D * heads per visible (query token, key) pair: QK^T and PV."""
    return sum(4 * w.head_dim * w.heads * visible(w, int(p))[1] for p in positions)


def measured_tensor_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def cpu_oracle_prefill_rate(w, host, budget_s, max_tokens=None, seed=0):
    """The oracle's prefill on random samples of the packed tokens (each call
    writes and attends its sample) for about budget_s; returns
    (TFLOP/s, seconds, description, tokens)."""
    import numpy as np
    import oracle
    P = len(host["positions"])
    shape = oracle.make_shape(w.rows, w.heads, w.kv_heads, w.head_dim, w.pages_per_row, host["k_pool"].shape[0],
                              oracle.BF16, window=w.window, rope_theta=w.rope_theta)
    rng = np.random.default_rng(seed)
    flops, spent, tokens = 0, 0.0, 0
    while True:
        idx = np.sort(rng.choice(P, 8, replace=False))
        sub = {k: np.ascontiguousarray(host[k][idx]) for k in ("q", "k_new", "v_new", "positions", "rows", "slots")}
        t0 = time.perf_counter()
        _, _, _, rc = oracle.prefill_paged(shape, sub["q"], sub["k_new"], sub["v_new"], sub["positions"],
                                           sub["rows"], sub["slots"], host["table"], host["k_pool"], host["v_pool"])
        spent += time.perf_counter() - t0
        assert rc == 0
        flops += prefill_flops(w, sub["positions"])
        tokens += len(idx)
        if (max_tokens and tokens >= max_tokens) or (not max_tokens and spent >= budget_s):
            break
    desc = f"oracle prefill of {tokens} tokens sampled at random from the {P} (8 per call), single thread"
    return flops / spent / 1e12, spent, desc, tokens


def run_prefill(args, w, world, rank, local, light=False):
    """Whole prefill calls timed (value), the attention kernel alone (roofline),
    end to end through pinned host buffers and the oracle; `light` keeps the
    first two (a per-config entry of the decode line)."""
    from paged_gqa_decode_step_gb300 import build
    build.build()
    from paged_gqa_decode_step_gb300 import binding as b

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    t = wl.generate_prefill(w, dev, seed=rank_seed(w, rank))
    P = w.tokens
    pos_list = t["positions"].cpu().tolist()
    num_pages = t["k_pool"].shape[0]
    cos, sin = b.rope_tables(w.rope_theta, w.head_dim, w.max_seq, torch.bfloat16)
    p = b.make_params(w.rows, w.heads, w.kv_heads, w.head_dim, w.pages_per_row, num_pages, torch.bfloat16,
                      window=w.window, rope_cos=cos, rope_sin=sin)
    ws = b.new_prefill_workspace(p, P)
    out = torch.empty_like(t["q"])
    flops = prefill_flops(w, pos_list)
    flush = torch.empty(4 * L2_BYTES // 4, dtype=torch.int32, device=dev)
    names = ("q", "k_new", "v_new", "positions", "rows", "slots", "table", "k_pool", "v_pool")

    def step():
        b.prefill_paged(p, *(t[k] for k in names), out, ws)

    for _ in range(args.warmup):
        step()
    b.check_status(ws)
    launches_per_step = b.last_launch_count()

    with ClockSampler(dev) as clocks:
        t_load = time.time()
        if not args.quick:
            keep_busy(step, 0.3, flush)
        barrier(world)
        ms = device_ms(step, args.steps, flush)
        t_end = time.time()
        barrier(world)
    clk = clocks.window(t_load, t_end)
    b.check_status(ws)
    if args.quick:
        if rank == 0:
            print(json.dumps({"quick": True, "workload": w.name, "ms_per_step": ms,
                              "tflops": flops / (ms * 1e-3) / 1e12}), flush=True)
        return None
    ms = max_over_ranks(ms, world)
    all_flops = sum_over_ranks(flops, world)
    value = all_flops / (ms * 1e-3) / 1e12

    # roofline: the attention kernel alone (prefill_attend), events around each launch
    att_ms = device_ms(lambda: b.prefill_attend(p, t["positions"], t["table"], t["k_pool"], t["v_pool"], out, ws),
                       max(20, min(args.steps, 200)), flush)
    b.check_status(ws)
    peak, peak_kind = measured_tensor_peak()
    achieved = flops / (att_ms * 1e-3) / 1e12
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "traffic": None, "kernel": f"prefill_kernel<{w.head_dim}>",
            "flops_per_launch": flops, "launch_us": att_ms * 1e3, "peak_kind": peak_kind}
    if light:
        return {"metric": PREFILL_METRIC, "value": value, "unit": "TFLOP/s", "ms_per_step": ms,
                "steps": args.steps, "tokens": P, "flops_per_step": flops,
                "frac_of_tensor_peak": value / world / peak, "roofline": roof,
                "l2": "L2 flushed (512 MB write) between timed calls, outside the events", "clocks": clk}

    # end to end: pinned host inputs in, output back, every call
    e2e_s, h2d, d2h = e2e_pipelined(
        t, ("q", "k_new", "v_new", "positions", "rows", "slots", "table"),
        lambda d, o: b.prefill_paged(p, d["q"], d["k_new"], d["v_new"], d["positions"], d["rows"], d["slots"],
                                     d["table"], t["k_pool"], t["v_pool"], o, ws),
        out, max(10, min(args.steps, 100)), world)
    e2e_s = max_over_ranks(e2e_s, world)
    b.check_status(ws)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host = {k: wl.to_numpy(v) for k, v in t.items()}
        rate, spent, desc, _ = cpu_oracle_prefill_rate(w, host, args.cpu_baseline_seconds)
        cpu = {"value": rate, "unit": "TFLOP/s", "cores": 1, "kind": "oracle", "sample": desc,
               "seconds": round(spent, 2), "cpu": cpu_model()}
    if rank != 0:
        return None
    return {
        "metric": PREFILL_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/k/v and prefilled pool, shuffled page table)",
        "config": {
            "workload": w.name, "rows_per_gpu": w.rows, "tokens_per_gpu": P, "prefix": list(w.prefix),
            "chunk": list(w.chunk), "heads": w.heads, "kv_heads": w.kv_heads, "head_dim": w.head_dim,
            "page_size": 64, "window": w.window, "rope_theta": w.rope_theta, "flops_per_step_per_gpu": flops,
            "l2": "L2 flushed (512 MB write) between timed steps, outside the events",
            "parallelism": f"replicas x{world} (rows sharded across ranks, no exchange)",
        },
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": all_flops / e2e_s / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }


def run_prefill_reference(args, w, world, rank):
    if rank != 0:
        return None
    t = wl.generate_prefill(w, "cpu", seed=rank_seed(w, 0))
    host = {k: wl.to_numpy(v) for k, v in t.items()}
    del t
    per_step = max(8, int(min(5.0, 90.0 / max(1, args.steps + args.warmup)) / 0.05) // 8 * 8)
    if args.warmup:
        cpu_oracle_prefill_rate(w, host, 0, max_tokens=8 * args.warmup, seed=1)
    rates = []
    spent_all, toks = 0.0, 0
    for k in range(max(1, args.steps)):
        r, spent, desc, n = cpu_oracle_prefill_rate(w, host, 0, max_tokens=per_step, seed=2 + k)
        rates.append(r)
        spent_all += spent
        toks += n
    rate = sum(rates) / len(rates)
    desc = f"oracle prefill of {toks} tokens sampled at random from the {w.tokens} (8 per call), single thread"
    return {
        "metric": PREFILL_METRIC, "value": rate, "unit": "TFLOP/s", "n_gpus": world, "steps": len(rates),
        "warmup": args.warmup, "ms_per_step": spent_all / len(rates) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "impl": "reference",
        "config": {"workload": w.name, "tokens_per_step": per_step, "tokens": w.tokens},
        "cpu_baseline": {"kind": "oracle", "cores": 1, "sample": desc, "value": rate, "unit": "TFLOP/s",
                         "cpu": cpu_model()},
        "e2e": {"value": rate, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------- packed --
PACKED_METRIC = "packed-sequence attention TFLOP/s (% of GB300 bf16 tensor peak)"


def packed_flops(w, positions):
    """4 * D * heads per visible (query, key) pair; sequences start at position 0."""
    return sum(4 * w.head_dim * w.heads * (min(int(p) + 1, w.window) if w.window > 0 else int(p) + 1)
               for p in positions)


def cpu_oracle_packed_rate(w, host, budget_s, max_seqs=None):
    """The oracle's packed attention on whole sequences of the row, shortest
    first, for about budget_s; returns (TFLOP/s, seconds, description, sequences)."""
    import numpy as np
    import oracle
    shape = oracle.make_shape(0, w.heads, w.kv_heads, w.head_dim, 1, 1, oracle.BF16, window=w.window,
                              rope_theta=w.rope_theta)
    starts = np.concatenate([[0], np.cumsum(w.lengths)])
    flops, spent, done = 0, 0.0, 0
    for s in np.argsort(w.lengths):
        lo, hi = starts[s], starts[s + 1]
        sub = {k: np.ascontiguousarray(host[k][lo:hi]) for k in ("q", "k", "v", "positions", "segments")}
        t0 = time.perf_counter()
        _, _, _, _, rc = oracle.packed(shape, sub["q"], sub["k"], sub["v"], sub["positions"], sub["segments"])
        spent += time.perf_counter() - t0
        assert rc == 0
        flops += packed_flops(w, sub["positions"])
        done += 1
        if (max_seqs and done >= max_seqs) or (not max_seqs and spent >= budget_s):
            break
    desc = f"oracle packed attention of the {done} shortest of {len(w.lengths)} sequences, single thread"
    return flops / spent / 1e12, spent, desc, done


def run_packed(args, w, world, rank, local, light=False):
    """As run_prefill, for sequences packed into one row."""
    from paged_gqa_decode_step_gb300 import build
    build.build()
    from paged_gqa_decode_step_gb300 import binding as b

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    t = wl.generate_packed(w, dev, seed=rank_seed(w, rank))
    P = w.tokens
    pos_list = t["positions"].cpu().tolist()
    cos, sin = b.rope_tables(w.rope_theta, w.head_dim, w.max_seq, torch.bfloat16)
    p = b.make_params(1, w.heads, w.kv_heads, w.head_dim, 1, 1, torch.bfloat16, window=w.window, rope_cos=cos,
                      rope_sin=sin)
    ws = b.new_packed_workspace(p, P)
    out = torch.empty_like(t["q"])
    flops = packed_flops(w, pos_list)
    flush = torch.empty(4 * L2_BYTES // 4, dtype=torch.int32, device=dev)
    names = ("q", "k", "v", "positions", "segments")

    def step():
        b.packed(p, *(t[k] for k in names), out, ws)

    for _ in range(args.warmup):
        step()
    b.check_status(ws)
    launches_per_step = b.last_launch_count()

    with ClockSampler(dev) as clocks:
        t_load = time.time()
        if not args.quick:
            keep_busy(step, 0.3, flush)
        barrier(world)
        ms = device_ms(step, args.steps, flush)
        t_end = time.time()
        barrier(world)
    clk = clocks.window(t_load, t_end)
    b.check_status(ws)
    if args.quick:
        if rank == 0:
            print(json.dumps({"quick": True, "workload": w.name, "ms_per_step": ms,
                              "tflops": flops / (ms * 1e-3) / 1e12}), flush=True)
        return None
    ms = max_over_ranks(ms, world)
    all_flops = sum_over_ranks(flops, world)
    value = all_flops / (ms * 1e-3) / 1e12

    att_ms = device_ms(lambda: b.packed_attend(p, t["v"], t["positions"], out, ws), max(20, min(args.steps, 200)),
                       flush)
    b.check_status(ws)
    peak, peak_kind = measured_tensor_peak()
    achieved = flops / (att_ms * 1e-3) / 1e12
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "traffic": None, "kernel": f"prefill_kernel<{w.head_dim},packed>",
            "flops_per_launch": flops, "launch_us": att_ms * 1e3, "peak_kind": peak_kind}
    if light:
        return {"metric": PACKED_METRIC, "value": value, "unit": "TFLOP/s", "ms_per_step": ms,
                "steps": args.steps, "tokens": P, "flops_per_step": flops,
                "frac_of_tensor_peak": value / world / peak, "roofline": roof,
                "l2": "L2 flushed (512 MB write) between timed calls, outside the events", "clocks": clk}

    e2e_s, h2d, d2h = e2e_pipelined(t, names, lambda d, o: b.packed(p, *(d[k] for k in names), o, ws), out,
                                    max(10, min(args.steps, 100)), world)
    e2e_s = max_over_ranks(e2e_s, world)
    b.check_status(ws)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host = {k: wl.to_numpy(v) for k, v in t.items()}
        rate, spent, desc, _ = cpu_oracle_packed_rate(w, host, args.cpu_baseline_seconds)
        cpu = {"value": rate, "unit": "TFLOP/s", "cores": 1, "kind": "oracle", "sample": desc,
               "seconds": round(spent, 2), "cpu": cpu_model()}
    if rank != 0:
        return None
    return {
        "metric": PACKED_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) q/k/v)",
        "config": {
            "workload": w.name, "tokens_per_gpu": P, "lengths": list(w.lengths), "heads": w.heads,
            "kv_heads": w.kv_heads, "head_dim": w.head_dim, "window": w.window, "rope_theta": w.rope_theta,
            "flops_per_step_per_gpu": flops,
            "l2": "L2 flushed (512 MB write) between timed steps, outside the events",
            "parallelism": f"replicas x{world} (rows sharded across ranks, no exchange)",
        },
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": all_flops / e2e_s / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }


def run_packed_reference(args, w, world, rank):
    if rank != 0:
        return None
    t = wl.generate_packed(w, "cpu", seed=rank_seed(w, 0))
    host = {k: wl.to_numpy(v) for k, v in t.items()}
    del t
    rates, spent_all, seqs = [], 0.0, 0
    for _ in range(max(1, args.steps)):
        r, spent, desc, n = cpu_oracle_packed_rate(w, host, 0, max_seqs=2)
        rates.append(r)
        spent_all += spent
        seqs += n
    rate = sum(rates) / len(rates)
    return {
        "metric": PACKED_METRIC, "value": rate, "unit": "TFLOP/s", "n_gpus": world, "steps": len(rates),
        "warmup": args.warmup, "ms_per_step": spent_all / len(rates) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "impl": "reference",
        "config": {"workload": w.name, "sequences_per_step": 2, "tokens": w.tokens},
        "cpu_baseline": {"kind": "oracle", "cores": 1, "sample": desc, "value": rate, "unit": "TFLOP/s",
                         "cpu": cpu_model()},
        "e2e": {"value": rate, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama8b_serving",
                    choices=sorted(wl.WORKLOADS) + sorted(wl.PREFILL_WORKLOADS) + sorted(wl.PACKED_WORKLOADS))
    ap.add_argument("--cpu-baseline-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--chunk-pages", type=int, default=0,
                    help="pages per split (0: the planner chooses)")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the per-config entries of the other workloads")
    ap.add_argument("--quick", action="store_true",
                    help="warm-up and timed steps only, no JSON line (for profiler captures)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.workload in wl.PREFILL_WORKLOADS or args.workload in wl.PACKED_WORKLOADS:
        if args.workload in wl.PREFILL_WORKLOADS:
            w = wl.PREFILL_WORKLOADS[args.workload]
            ref, ours = run_prefill_reference, run_prefill
        else:
            w = wl.PACKED_WORKLOADS[args.workload]
            ref, ours = run_packed_reference, run_packed
        if args.impl == "reference":
            line = ref(args, w, world, rank)
        else:
            line = ours(args, w, world, rank, local)
        if line is not None:
            print(json.dumps(line), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    w = wl.WORKLOADS[args.workload]
    if args.impl == "reference":
        line = run_reference(args, w, world, rank)
    else:
        line = run_ours(args, w, world, rank, local)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
