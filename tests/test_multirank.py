"""Host logic of the multi-rank benchmark (replicas, one frame per rank, weak
scaling) with world size 2 over gloo on CPU: the job's time is the slowest
rank's, its throughput counts every rank's pixels."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [2.0 + rank, 1.0 + 3 * rank]  # rank 1 is slower in both
        out = bench.max_over_ranks(ms, dist, "cpu")
        q.put((rank, out, bench.job_throughput(world, 1920 * 1080, out[0])))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_throughput_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, out, thr in res:
        assert out == [3.0, 4.0]
        assert abs(thr - 2 * 1920 * 1080 / 1e6 / 3e-3) < 1e-6


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert abs(bench.job_throughput(1, 1e6, 1.0) - 1000.0) < 1e-9
