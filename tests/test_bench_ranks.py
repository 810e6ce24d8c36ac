"""The multi-rank bench logic on CPU with gloo (world size 2): every rank gets the
slowest rank's time, and the whole-job rate counts the units of all replicas."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = [3.0, 7.5][rank]
    slowest = bench.max_over_ranks(mine, dist, "cpu")
    rate = bench.whole_job_rate(100.0, world, slowest)
    q.put((rank, slowest, rate))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [7.5, 7.5]
    assert got[0][2] == pytest.approx(2 * 100.0 / 7.5e-3)


def test_single_rank_needs_no_group():
    assert bench.max_over_ranks(4.25) == 4.25
    assert bench.whole_job_rate(10.0, 1, 2.0) == pytest.approx(5000.0)
