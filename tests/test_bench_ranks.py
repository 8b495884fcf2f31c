"""The benchmark's multi-rank host logic on CPU: two gloo ranks (127.0.0.1),
max over ranks of the per-rank timings, the whole-job weak-scaling rate,
and the reference arm doing its work on rank 0 only."""
import os
import socket
import types

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r measured (r + 1) ms on leg A and (10 - r) ms on leg B
        got = bench.max_over_ranks([rank + 1.0, 10.0 - rank], world)
        results[rank] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), results), nprocs=world, join=True)
        got = dict(results)
    assert got[0] == [2.0, 10.0] and got[1] == [2.0, 10.0]


def test_max_over_ranks_single_rank_is_identity():
    assert bench.max_over_ranks([3, 4.5], 1) == [3.0, 4.5]


def test_whole_job_rate_is_weak_scaling():
    # two ranks each processing 1e9 bytes, slowest rank 2 ms -> 1e12 B/s
    assert bench.whole_job_rate(1e9, 2, 2.0) == pytest.approx(1e12)
    assert bench.whole_job_rate(1e9, 1, 1.0) == pytest.approx(1e12)


def test_reference_arm_runs_on_rank_zero_only():
    args = types.SimpleNamespace(steps=1, warmup=3, cpu_budget=1.0)
    assert bench.run_reference(args, rank=1, world=2) is None
