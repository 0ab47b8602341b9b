"""The multi-process host logic of bench.py on CPU: two gloo ranks (replicas,
no collective on the data path) combine their step times by the maximum and
report the whole-job throughput of both replicas."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank                        # rank 1 is the slow one
        slowest = bench.max_over_ranks(ms, world, "cpu")
        dist.barrier()
        out.put((rank, slowest, bench.whole_job_tflops(world, 1e12, 4, slowest)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [15.0, 15.0]
    # two replicas of 1e12 FLOP per step, 4 steps in 15 ms
    assert got[0][2] == pytest.approx(2 * 1e12 * 4 / 15e-3 / 1e12)


def test_single_rank_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.whole_job_tflops(1, 2e12, 10, 20.0) == pytest.approx(1000.0)
