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


def _legs_rank_main(rank, world, port, results):
    # the rank logic of the GPU bench with host-timed stand-in legs: rank r's
    # leg "a" sleeps (r + 1) * 5 ms and leg "b" 5 ms; timing, max over ranks
    # and the summary run exactly as in run_ours
    import time as _t
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        legs = [("a", lambda: _t.sleep((rank + 1) * 5e-3)), ("b", lambda: _t.sleep(5e-3))]
        ms, (t0, t1) = bench.time_legs(legs, 4, 3, bench.HostTimer(), barrier=dist.barrier)
        names = list(ms)
        ms = dict(zip(names, bench.max_over_ranks([ms[n] for n in names], world)))
        meta = {"a": dict(bytes=1e9, flops=2e12, bound="tensor", dtype="f16", kernel=None),
                "b": dict(bytes=5e8, flops=0, bound="hbm", dtype="u8", kernel=None)}
        line = bench.summarize(ms, meta, world, {"hbm_gbs": 1000.0, "bf16_tflops": 100.0}, "test", headline="a")
        results[rank] = (ms, line, t1 - t0)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_bench_rank_logic_two_gloo_ranks():
    world = 2
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_legs_rank_main, args=(world, _free_port(), results), nprocs=world, join=True)
        got = dict(results)
    ms0, line0, wall = got[0]
    assert got[1][0] == ms0  # both ranks hold the max over ranks
    assert ms0["a"] == pytest.approx(10.0, rel=0.5) and ms0["a"] > ms0["b"]  # rank 1's slower leg
    # whole-job rates: both ranks' bytes over the slowest rank's time
    assert line0["value"] == pytest.approx(2 * 1e9 / (ms0["a"] * 1e-3) / 1e9)
    a = line0["legs"]["a"]
    assert a["tflops"] == pytest.approx(2 * 2e12 / (ms0["a"] * 1e-3) / 1e12)
    # roofline fractions are per GPU
    assert a["roofline"]["frac"] == pytest.approx(a["tflops"] / 2 / 100.0)
    assert line0["legs"]["b"]["roofline"]["bound"] == "hbm"
    assert line0["roofline"]["kernel"] == "a"  # the longest leg dominates
    assert line0["ms_per_step"] == pytest.approx(ms0["a"] + ms0["b"])
    assert wall >= 4 * (ms0["b"] * 1e-3)


def test_clock_samples_filtered_to_the_timed_window():
    import datetime
    def row(sec, mhz, cap="Not Active"):
        ts = datetime.datetime(2026, 1, 2, 3, 4, 5) + datetime.timedelta(seconds=sec)
        return f"{ts.strftime('%Y/%m/%d %H:%M:%S.%f')[:-3]}, 0, {mhz}, 2070, 900.0, 0x0, Not Active, " \
               f"Not Active, Not Active, {cap}"
    lines = [row(0, 1000), row(1, 2070), row(1.5, 2060, "Active"), row(2, 2050), row(9, 500)]
    base = datetime.datetime(2026, 1, 2, 3, 4, 5).timestamp()
    c = bench.summarize_clocks(lines, base + 0.9, base + 2.1)
    assert c["samples"] == 3 and c["sm_mhz"] == 2060 and c["reasons"] == ["sw_power_cap"]
    assert bench.summarize_clocks(lines, base + 3, base + 4)["reasons"] == ["unsampled"]


def test_gpus_flag_must_match_world_size(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setenv("RANK", "0")
    assert bench.main(["--gpus", "2", "--no-cpu-baseline"]) == 2
