"""The benchmark's multi-rank bookkeeping on CPU ranks (gloo, world size 2).

`bench.py --gpus N` runs N independent replicas of the draft step (the step
does not shard): the ranks meet at a barrier, the slowest rank's time is the
job's time, and rank 0 reports the steps of all ranks over it.  The reference
arm runs on rank 0 alone.
"""

from __future__ import annotations

import argparse
import multiprocessing as mp
import os
import socket

import pytest


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, local_ms, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        slowest = bench.barrier_max(world, local_ms[rank], device="cpu")
        q.put((rank, slowest, bench.job_value(world, 10, slowest)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_report_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    local_ms = [120.0, 150.0]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, local_ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        results = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [p.exitcode for p in procs] == [0, 0]
    assert [r for r, _, _ in results] == [0, 1]
    for _, slowest, value in results:
        assert slowest == 150.0                          # every rank sees the max
        assert value == pytest.approx(2 * 10 / 0.150)    # all ranks' steps over it


def test_job_value_single_rank():
    import bench
    assert bench.barrier_max(1, 42.0) == 42.0            # no collective for one rank
    assert bench.job_value(1, 200, 40.0) == pytest.approx(5000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    args = argparse.Namespace(config="qwen_dense", steps=3, warmup=3, gpus=2)
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""
