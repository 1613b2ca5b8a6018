"""The multi-rank timing logic of bench.py on CPU: two gloo ranks, each with
its own step time; every rank sees the maximum, and the whole-job rate counts
the tokens of both ranks over the slowest rank's time."""
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


def _worker(rank, world, port, out):
    import sys
    import torch.distributed as dist
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = bench.reduce_max(1.5 + rank, "cpu")
    out[rank] = (ms, bench.whole_job_rate(4096, world, ms))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_rate():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0][0] == out[1][0] == 2.5
    assert out[0][1] == pytest.approx(2 * 4096 / 2.5e-3)


def test_single_process_no_group():
    import bench
    assert bench.reduce_max(3.0, "cpu") == 3.0
    assert bench.whole_job_rate(100, 1, 1.0) == pytest.approx(1e5)
