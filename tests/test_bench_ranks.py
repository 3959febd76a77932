"""The replicas path of bench.py on CPU: two gloo ranks (world size 2), each with its own timed
region; the job's time is the slowest rank's (all-reduce MAX) and the whole-job throughput is
the steps of every rank over that time."""
import os
import socket

import pytest
import torch.multiprocessing as mp

pytestmark = pytest.mark.cpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import sys

    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.rank_max_ms(10.0 + 5.0 * rank, world, "cpu")      # rank 1 is the slower one
        out[rank] = (ms, bench.job_steps_per_s(world, 100, ms))
    finally:
        dist.destroy_process_group()


def test_job_time_is_the_slowest_rank_and_throughput_counts_every_rank():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        ms, v = out[r]
        assert ms == 15.0
        assert v == pytest.approx(2 * 100 / 0.015)


def test_one_rank_keeps_its_own_time():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.rank_max_ms(12.5, 1, "cpu") == 12.5
    assert bench.job_steps_per_s(1, 400, 1.5) == pytest.approx(400 / 1.5e-3)
