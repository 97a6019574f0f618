"""The multi-rank logic of bench.py on CPU: two gloo ranks (replicas) agree
on the slowest rank's time and rank 0's aggregate counts both replicas."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        bench.barrier()
        local_ms = [12.5, 20.0][rank]                 # rank 1 is the slow one
        ms = bench.max_over_ranks(local_ms)
        out[rank] = (ms, bench.whole_job_tflops(world, 2e9, 100, ms))
        bench.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time_and_sum_the_work():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 20.0
    # 2 replicas x 100 steps x 2 GFLOP in 20 ms = 20 TFLOP/s
    assert res[0][1] == pytest.approx(20.0)


def test_single_process_passthrough():
    import bench
    assert not dist.is_initialized()
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_tflops(1, 1e12, 1, 1000.0) == pytest.approx(1.0)
