"""World-size-2 test of the benchmark's multi-rank host logic on CPU ranks (gloo).

The path shards by sequence with no exchange step, so N GPUs run N replicas: each rank
times its own steps between barriers, every timing is reduced by its maximum over the
ranks (the job is as fast as its slowest rank), and the whole-job throughput counts the
sequences of every rank.  No GPU is involved.
"""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        timings = [1.0 + rank, 5.0 - rank, 2.5 + 0.25 * rank]     # this rank's step timings
        got = bench.max_over_ranks(dist, timings, "cpu")
        dist.barrier()
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [2.0, 5.0, 2.75]
    sys.path.insert(0, ROOT)
    import bench
    # 32 sequences per rank, 2 ranks, 0.1 ms per step -> 640,000 tokens/s for the job
    assert bench.job_throughput(32, 2, 0.1) == pytest.approx(640000.0)
    assert bench.max_over_ranks(None, [3, 1.5], "cpu") == [3.0, 1.5]
