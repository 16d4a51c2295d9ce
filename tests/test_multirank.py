"""The benchmark's multi-rank host logic on CPU: two gloo ranks, each timing its own workload
instance; the job's step time is the slowest rank's and the value counts every rank's work."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 2.0 + rank  # rank 1 is the slow one
    out[rank] = bench.ranks_max(ms, dist, "cpu")
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_job_value():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        assert out[0] == out[1] == 3.0
    import bench

    assert bench.job_value(2, 1e12, 1000.0) == pytest.approx(2.0)
