"""The multi-rank path of bench.py (replicas: no collective on the data path, max over
ranks for the time) on CPU with two gloo ranks."""

import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = [2.0, 5.0][rank]
        ms_max = bench.reduce_max(ms, torch.device("cpu"))
        out[rank] = (ms_max, bench.whole_job_tflops(1e12, ms_max, world))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_whole_job_value():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        ms_max, value = out[r]
        assert ms_max == 5.0
        assert abs(value - world * 1e12 / 5e-3 / 1e12) < 1e-9


def test_single_process_identity():
    import bench
    assert bench.reduce_max(3.5, torch.device("cpu")) == 3.5
    assert abs(bench.whole_job_tflops(2e12, 4.0, 1) - 500.0) < 1e-9
