"""The multi-GPU benchmark path runs independent replicas (the tail has no cross-GPU
exchange); its only collective is the max-over-ranks of the timed region.  Exercised
here with two gloo ranks on the CPU."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed = [12.5, 30.0][rank]  # rank 1 is the slow one
    m = bench.max_over_ranks(elapsed)
    us = bench.job_us_per_call(m, steps=100, world=world)
    q.put((rank, m, us))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_count_all_calls():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, us in got:
        assert m == 30.0
        assert us == pytest.approx(30.0 * 1000 / 200)


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_us_per_call(10.0, 10, 1) == pytest.approx(1000.0)
