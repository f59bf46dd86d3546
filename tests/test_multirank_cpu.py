"""The bench's N > 1 path on the CPU: two ``gloo`` ranks exercise the barrier,
the max over ranks (the slowest rank's time) and the whole-job rate, and the
reference arm's rank rule (rank 0 alone runs; other ranks return without
work).  The replicas share no data, so these host steps are the whole of the
multi-rank logic.
"""
import argparse
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench._barrier(world)
        ms = bench._max_over_ranks(1.25 + rank, world)          # rank r "took" 1.25 + r ms
        rate = bench._whole_job_rate(32768, world, ms)
        ns = argparse.Namespace(steps=1, warmup=0)
        ref = bench.run_reference(ns, rank, world) if rank != 0 else "rank0"
        bench._barrier(world)
        q.put((rank, ms, rate, ref))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_barrier_max_and_rate():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    try:
        out = sorted(q.get(timeout=120) for _ in range(world))
    finally:
        for p in procs:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    for rank, ms, rate, ref in out:
        assert ms == pytest.approx(2.25)                         # every rank sees the slowest rank's time
        assert rate == pytest.approx(2 * 32768 / 2.25e-3)        # both ranks' tokens over that time
        if rank != 0:
            assert ref is None                                   # reference arm: rank 0 alone runs


def test_single_rank_helpers_need_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    bench._barrier(1)
    assert bench._max_over_ranks(3.5, 1) == 3.5
    assert bench._whole_job_rate(32768, 1, 2.0) == pytest.approx(32768 / 2e-3)


def test_rotation_rate_arithmetic():
    """The bench's tensor-rate line: terms x 2 d^2 flops per vector over the launch time."""
    sys.path.insert(0, ROOT)
    import bench

    r = bench._rotation_rate(1000, 2, 4, 3, 1.0, 100.0)        # 3 * 2 * 16 * 2000 flops in 1 ms
    assert r["executed_tflops"] == pytest.approx(3 * 2 * 16 * 2000 / 1e-3 / 1e12, abs=0.05)
    assert r["algorithmic_tflops"] == pytest.approx(r["executed_tflops"] / 3, abs=0.05)
    r = bench._rotation_rate(32768, 8, 128, 3, 0.0349, 1810.1)
    assert r["frac_executed"] == pytest.approx(r["executed_tflops"] / 1810.1, rel=1e-3)
