"""bench.py's multi-rank logic on CPU: two gloo ranks (one process each, as torchrun launches them)
agree on the slowest rank's step time, and the whole-job rate counts every rank's units. The
reference arm does no work on ranks other than 0."""
import argparse
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


def _rank_main(rank, world, port, times, results):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], dist, "cpu")
        results.put((rank, ms, bench.job_rate(world, 64, ms)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, times = 2, [0.5, 0.8]
    ctx = mp.get_context("spawn")
    results = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(results.get(timeout=10) for _ in range(world))
    for rank, ms, rate in got:
        assert ms == max(times)
        assert rate == pytest.approx(world * 64 / (max(times) * 1e-3))


def test_single_rank_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.25, None, "cpu") == 1.25
    assert bench.job_rate(1, 64, 1.0) == pytest.approx(64000.0)


def test_reference_arm_only_runs_on_rank_0():
    sys.path.insert(0, ROOT)
    import bench
    args = argparse.Namespace(steps=1, warmup=0)
    assert bench.reference_arm(args, world=2, rank=1) is None   # returns before touching CUDA
