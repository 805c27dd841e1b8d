"""The host side of the multi-rank benchmark, run as two gloo ranks on the CPU: the
slowest rank's times are the job's, the throughput counts every rank's rows, and under a
multi-rank launch the oracle arm runs on rank 0 only."""

import io
import os
import socket
import contextlib

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r measured (1 + r, 10 - r, 0.5 r): every rank must see the maxima
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 0.5 * rank], torch.device("cpu"))
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    results = dict(q.get(timeout=5) for _ in range(world))
    for r in range(world):
        assert results[r] == [2.0, 10.0, 0.5]


def test_whole_job_throughput_counts_every_rank():
    assert bench.rows_per_second(32, 1, 0.1) == pytest.approx(320000.0)
    assert bench.rows_per_second(32, 4, 0.1) == pytest.approx(4 * 320000.0)


def test_reference_arm_runs_on_rank_zero_only():
    class Args:
        workload = "tiny"
        warmup = 3
        steps = 1
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        bench.run_reference(Args(), rank=1, world=2)
    assert out.getvalue() == ""
