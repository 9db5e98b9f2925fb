"""The multi-rank bench path on CPU: two gloo ranks run the slowest-rank
reduction and the whole-job throughput formula that bench.py uses under
torchrun (no GPU, no data-path collective)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        t = bench.max_over_ranks(times[rank], world, torch.device("cpu"))
        v = bench.whole_job_tflops(2.0 * 4096 * 4096 * 7168, 10, world, t)
        out[rank] = (t, v)
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world = 2
    times = [1.25, 3.5]
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), times, out), nprocs=world,
                           start_method="spawn", join=True)
        res = dict(out)
    flops = 2.0 * 4096 * 4096 * 7168
    for r in range(world):
        t, v = res[r]
        assert t == max(times)
        assert v == pytest.approx(world * flops * 10 / (max(times) * 1e-3) / 1e12)


def test_one_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.0, 1, torch.device("cpu")) == 2.0
    assert bench.whole_job_tflops(1e12, 1, 1, 1000.0) == pytest.approx(1.0)
