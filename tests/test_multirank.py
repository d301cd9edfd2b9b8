"""The multi-process logic of bench.py on CPU: two gloo ranks.

The path shards along N without any data exchange, and every box here has one GPU, so
`bench.py --gpus N` runs one replica per rank (weak scaling). What the ranks share is the timing:
a barrier around the timed region and the maximum over ranks of its length, and the whole-job
rate (per-rank work x ranks / slowest time). Both are checked here with a real gloo process group.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, times, out):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = bench.max_over_ranks(times[rank], dist, torch.device("cpu"))
        step_s = ms / 1e3 / 10
        rate = bench.job_rate(28_210_688, step_s, world)
        out[rank] = (ms, rate)
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_is_the_slowest_rank():
    world, port = 2, _free_port()
    times = [3.25, 4.75]          # milliseconds of the timed region on each rank
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    assert set(res) == {0, 1}
    for rank in range(world):
        ms, rate = res[rank]
        assert ms == max(times)                             # every rank reports the slowest rank's time
        assert rate == pytest.approx(2 * 28_210_688 / (4.75e-3 / 10))   # both replicas' work / that time


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(1.5, None, torch.device("cpu")) == 1.5
    assert bench.job_rate(100.0, 2.0, 1) == 50.0
