"""The multi-rank host logic of bench.py on CPU: two gloo ranks (one process each, as torchrun
would launch them on two GPUs) agree on the slowest rank's time, and the whole-job throughput
counts every rank's units over that time."""
import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [1.5, 2.25][rank]              # the second rank is the slower one
        slowest = bench.max_over_ranks(ms, torch.device("cpu"))
        out[rank] = (slowest, bench.job_throughput(1000.0, world, slowest))
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
        res = dict(out)
    for rank in range(world):
        slowest, tput = res[rank]
        assert slowest == 2.25
        assert abs(tput - 2 * 1000.0 / 2.25e-3) < 1e-6


def test_single_rank_is_its_own_time():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.0, torch.device("cpu")) == 3.0
    assert bench.job_throughput(500.0, 1, 2.0) == 500.0 / 2e-3
