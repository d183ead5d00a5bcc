"""The N > 1 path of bench.py on CPU with world_size-2 gloo process groups.

The attention path has no cross-GPU exchange, so N GPUs run N independent
replicas.  What the ranks share is the timing: a barrier around the timed
region, the maximum of the per-rank times, the whole-job rate over it, and the
reference arm, which only rank 0 runs.  These tests run that host-side logic
in two processes.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        dist.barrier()
        local_ms = 100.0 + 50.0 * rank          # rank 1 is the slow one
        slowest = bench.max_over_ranks(local_ms, w, "cpu")
        rate = bench.job_rate(2.0e12, 10, w, slowest)
        dist.barrier()
        out.put((r, w, local, slowest, rate))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_sum_the_work():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(out.get(timeout=10) for _ in range(2))
    for rank, (r, w, local, slowest, rate) in enumerate(got):
        assert (r, w, local) == (rank, 2, rank)
        assert slowest == 150.0
        # 2 replicas x 10 steps x 2 TFLOP over 150 ms
        assert rate == pytest.approx(2 * 10 * 2.0e12 / 0.150 / 1e12)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(12.5, 1) == 12.5
    assert bench.job_rate(1.0e12, 4, 1, 1000.0) == pytest.approx(4.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import argparse

    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = argparse.Namespace(workload=bench.WORKLOAD, steps=1, warmup=0)
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""   # rank 1 does no work and prints nothing
