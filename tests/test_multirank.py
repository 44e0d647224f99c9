"""The benchmark's multi-rank host logic on CPU (gloo, world size 2):
replicas run independently, the job's time is the slowest rank's, and the
job's rate counts every rank's work (weak scaling)."""
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
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [3.0, 5.0][rank]                       # rank 1 is the slow one
    worst = bench.max_over_ranks(ms, world)
    rate = bench.whole_job_rate(1e9, world, worst)
    dist.barrier()
    q.put((rank, worst, rate))
    dist.destroy_process_group()


def test_two_rank_max_and_weak_scaling_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, worst, rate in out:
        assert worst == 5.0
        assert rate == pytest.approx(2 * 1e9 / 5e-3)


def test_single_rank_passthrough():
    import bench
    assert bench.max_over_ranks(1.5, 1) == 1.5
    assert bench.whole_job_rate(10.0, 1, 1000.0) == 10.0
