"""The N > 1 path of bench.py on CPU: two gloo ranks, each an independent
replica; the whole-job throughput divides all ranks' units by the slowest
rank's timed region (max over ranks), identically on every rank."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    local = 1.0 + rank  # rank 1 is the slow one
    value, t = bench.job_throughput(local, 100)
    q.put((rank, value, t))
    dist.barrier()
    dist.destroy_process_group()


def test_job_throughput_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, value, t in got:
        assert t == pytest.approx(2.0)            # the slowest rank's time
        assert value == pytest.approx(2 * 100 / 2.0)  # all ranks' units / that time


def test_job_throughput_single_process():
    sys.path.insert(0, ROOT)
    import bench

    value, t = bench.job_throughput(0.5, 64)
    assert t == 0.5 and value == 128.0
