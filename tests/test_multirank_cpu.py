"""The benchmark's multi-rank host logic on CPU (gloo, world size 2).

Each rank runs its own replica of the workload (no data-path collective);
only the timing is combined: the slowest rank's time sets the job time, and
the job throughput counts every rank's work.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, lr = bench.dist_env()
        assert (w, r, lr) == (world, rank, rank)
        bench.barrier(world)
        t = bench.max_over_ranks(1.5 + rank, world)     # rank 0: 1.5 ms, rank 1: 2.5 ms
        q.put((rank, t))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 2.5), (1, 2.5)]


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    bench.barrier(1)


def test_whole_job_value_counts_every_rank():
    import workloads
    w = workloads.WORKLOADS[workloads.BENCH_WORKLOAD]
    assert w.flops() == pytest.approx(4 * 2 * 32 * 4096 * 4096 * 128 / 2)
    ms = 0.25
    one = w.flops() / (ms * 1e-3) / 1e12
    four = w.flops() * 4 / (ms * 1e-3) / 1e12
    assert four == pytest.approx(4 * one)
