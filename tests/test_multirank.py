"""Two-rank (gloo, CPU) check of the bench's replica aggregation: every rank
learns the slowest rank's time, and the whole-job rate counts every rank's
steps over that time (weak scaling, no collective on the data path)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local = [0.5, 2.0][rank]
    m = bench.job_max(local, dist, "cpu")
    out[rank] = (m, bench.job_rate(100, world, m))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_rate():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        ps = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in ps:
            p.start()
        for p in ps:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0] == res[1] == (2.0, 100.0)


def test_single_process_aggregation_is_identity():
    import bench
    assert bench.job_max(1.25, None, "cpu") == 1.25
    assert bench.job_rate(10, 1, 0.5) == 20.0
