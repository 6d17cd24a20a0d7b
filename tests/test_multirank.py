"""The bench's multi-rank path, on CPU with gloo and two ranks.

Ranks shard rows (each draws its own seeded batch), exchange no data, and
combine only timings and byte counts: max over ranks for time, sum for bytes.
"""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench
    from paged_gqa_decode_step_gb300 import workloads as wl
    w_, r_, _ = bench.dist_setup()
    assert (w_, r_) == (world, rank)
    w = wl.TINY
    seed = bench.rank_seed(w, rank)
    t = wl.generate(w, "cpu", seed=seed)
    kvb = bench.kv_bytes(w, t["positions"].tolist())
    fake_ms = 1.0 + rank                       # rank 1 is the slow one
    bench.barrier(world)
    mx = bench.max_over_ranks(fake_ms, world)
    total = bench.sum_over_ranks(kvb, world)
    q.put((rank, seed, kvb, mx, total, t["q"].float().sum().item()))
    import torch.distributed as dist
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_ranks_shard_rows_and_reduce_timings():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=100) for _ in range(world))
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    (r0, s0, b0, m0, t0, q0), (r1, s1, b1, m1, t1, q1) = res
    assert s0 != s1 and q0 != q1                     # different rows on each rank
    assert m0 == m1 == 2.0                           # max over ranks
    assert t0 == t1 == b0 + b1                       # whole-job bytes
