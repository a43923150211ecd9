"""The N>1 host logic of bench.py on CPU: two gloo ranks, each timing an
independent replica; the job rate uses the slowest rank and counts both
ranks' work."""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        total_ms = [40.0, 50.0][rank]              # rank 1 is the slower replica
        slowest = bench.max_over_ranks(total_ms, world, "cpu")
        out[rank] = (slowest, bench.job_throughput(1e12, 10, slowest, world))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_reduction():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
        res = dict(out)
    assert res[0] == res[1]
    slowest, rate = res[0]
    assert slowest == 50.0
    # 2 ranks x 10 steps x 1e12 units over 50 ms = 400 (x1e12 units/s)
    assert abs(rate - 400.0) < 1e-9


def test_single_rank_is_identity():
    assert bench.max_over_ranks(12.5, 1, "cpu") == 12.5
    assert abs(bench.job_throughput(2e12, 4, 8.0, 1) - 1000.0) < 1e-9
