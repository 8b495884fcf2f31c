#!/usr/bin/env python
"""Benchmark of the MLA NVFP4 hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
  1. cache write: the 262,144 latent tokens of the DeepSeek-V3-shaped decode
     batch (64 x 4096) quantised into 432-byte records of a paged cache;
  2. decode: absorbed decode of that batch (64 sequences x 128 heads x 4096
     keys, 576-d bf16 queries, random page permutation, split-K + LSE merge);
  3. prefill: causal varlen prefill of 8 x 4096 tokens x 128 heads (q/k 192,
     v 128) with the fused NVFP4 output.
Legs are timed with CUDA events on the launching stream; L2 is flushed (a
256 MB write) before every leg.  `value` is the decode leg's algorithmic
HBM throughput (the metric's first part); the prefill TFLOP/s and the
cache-write GB/s are reported beside it.

--impl reference times the CPU oracle (test infrastructure) on a bounded
sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA NVFP4 decode HBM GB/s (% peak); prefill TFLOP/s with fused NVFP4 output"
UNIT = "GB/s"
WORKLOAD = ("decode_dsv3: B64 H128 L4096 paged 432B NVFP4 cache (cache write of its 262144 tokens + "
            "split-K decode) + prefill_8x4096: causal varlen H128 qk192 v128 fused NVFP4 out")
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
SM_COUNT, SM_MAX_MHZ, FP32_LANES = 152, 2070.0, 128


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def decode_bytes(w) -> int:
    """Algorithmic bytes of one decode: every attended record once, Q, out,
    the page table / indices and lengths."""
    rec = w.tokens_attended() * w.record_bytes
    q = w.q.numel() * 2
    out = w.batch * w.heads * 512 * 2
    idx = (w.page_table.numel() * 4 + w.batch * 4) if w.paged else w.topk_indices.numel() * 4
    return rec + q + out + idx


def decode_flops(w) -> float:
    return 2.0 * w.tokens_attended() * w.heads * (576 + 512)


def cache_write_bytes(w) -> int:
    T = w.kv_c.shape[0]
    return T * (512 * 2 + 64 * 2 + 8 + w.record_bytes)


def prefill_flops(p) -> float:
    import torch
    lens = (p.cu_seqlens[1:] - p.cu_seqlens[:-1]).to("cpu", torch.int64)
    pairs = int((lens * (lens + 1) // 2).sum())
    return 2.0 * pairs * p.heads * (192 + 128)


def prefill_bytes(p) -> int:
    T, H = p.total_tokens, p.heads
    return T * H * (192 * 2 * 2 + 128 * 2) + T * H * 64 + ((T + 127) // 128 * 128) * H * 8


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        # raw samples: $MLA_BENCH_CLOCKS_DIR/clocks_gpu<i>.csv when set (kept), else a temporary file
        keep = os.environ.get("MLA_BENCH_CLOCKS_DIR")
        self.temporary = not keep
        if keep:
            self.path = os.path.join(keep, f"clocks_gpu{gpu_index}.csv")
        else:
            fd, self.path = tempfile.mkstemp(prefix=f"mla_clocks_gpu{gpu_index}_", suffix=".csv")
            os.close(fd)

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        try:
            return self._summary()
        finally:
            if self.temporary and os.path.exists(self.path):
                os.remove(self.path)

    def _summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": ["unsampled"]}
        loaded = sorted(sm)[len(sm) // 4:] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax, "samples": len(sm),
                "reasons": sorted(reasons)}


def _traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was
    captured on the current source of that kernel."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel)
    if not d:
        return None
    src = os.path.join(ROOT, "mla_attention_nvfp4_gb300", "csrc", d["source"])
    if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != d["sha"]:
        return None
    return d["bytes_per_launch"]


def max_over_ranks(values, world, device=None):
    """Element-wise max of per-rank timings over the process group: the
    slowest rank sets the whole job's time.  NCCL reduces on the GPU, gloo
    (CPU tests) on the host."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    dev = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(units_per_rank, world, ms):
    """Weak scaling: every rank processes the same units (independent
    batches), so the job's rate is all ranks' units over the slowest rank's
    time in milliseconds."""
    return world * units_per_rank / (ms * 1e-3)


def run_ours(args, rank, world):
    import torch
    import mla_attention_nvfp4_gb300 as mla
    from mla_attention_nvfp4_gb300 import workloads

    torch.cuda.set_device(rank % max(1, torch.cuda.device_count()))
    dev = torch.device("cuda", torch.cuda.current_device())
    mla.load_library()
    peaks, peak_src = _peaks()
    stream = torch.cuda.current_stream()

    # --- workload (device-resident), seed 0 -----------------------------
    w = workloads.decode_dsv3(device=dev, batch=16 if args.case == "decode-steady" else 64)
    decode_splits = 1 if args.case == "decode-steady" else 0
    if args.case == "profile":
        # the same legs on a prefill of 2 x 4096 tokens (about 1.8 GB on the
        # device in all), for ncu captures; never a bench value
        p = workloads.prefill("prefill_2x4096", seq_lens=(4096, 4096), device=dev)
    else:
        p = workloads.prefill_8x4096(device=dev)
    gs = mla.mla_nvfp4_global_scale(w.kv_c)
    gsp = mla.mla_nvfp4_global_scale(p.v)
    cache = torch.zeros((w.num_slots, w.record_bytes), dtype=torch.uint8, device=dev)
    out = torch.empty((w.batch, w.heads, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.batch, w.heads), dtype=torch.float32, device=dev)
    ws = torch.empty(max(256, mla.mla_nvfp4_decode_workspace_size(w.batch, w.heads, decode_splits)), dtype=torch.uint8,
                     device=dev)
    codes = torch.empty((p.total_tokens, p.heads * 64), dtype=torch.uint8, device=dev)
    scales = torch.empty(mla.prefill_scale_bytes(p.total_tokens, p.heads), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def leg_cache_write():
        mla.mla_nvfp4_cache_write(w.kv_c, w.k_pe, w.slot_mapping, cache, gs, err)

    def leg_decode():
        mla.mla_nvfp4_decode(w.q, cache, gs, w.softmax_scale, page_table=w.page_table, seq_lens=w.seq_lens,
                             out=out, lse=lse, workspace=ws, error_word=err, num_splits=decode_splits)

    def leg_prefill():
        mla.mla_nvfp4_prefill_fused_out(p.q, p.k, p.v, p.cu_seqlens, p.max_seqlen, p.softmax_scale, gsp,
                                        out_codes=codes, out_scales=scales, error_word=err)

    legs = [("cache_write", leg_cache_write), ("decode", leg_decode), ("prefill", leg_prefill)]
    launches_per_step = mla.LAUNCHES_PER_CALL["cache_write"] + mla.decode_launches(w.batch, w.heads, decode_splits) + \
        mla.LAUNCHES_PER_CALL["prefill"]

    def step(record=None):
        for name, fn in legs:
            flush.zero_()
            if record is None:
                fn()
            else:
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                record[name].append((e0, e1))

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item()):#x} after warm-up")

    rec = {n: [] for n, _ in legs}
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        t0 = time.perf_counter()
        for _ in range(args.steps):
            step(rec)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    leg_ms = {n: sum(a.elapsed_time(b) for a, b in rec[n]) / args.steps for n in rec}
    step_ms = sum(leg_ms.values())
    step_ms, leg_ms["decode"], leg_ms["prefill"], leg_ms["cache_write"] = max_over_ranks(
        [step_ms, leg_ms["decode"], leg_ms["prefill"], leg_ms["cache_write"]], world, dev)

    dec_b, cw_b = decode_bytes(w), cache_write_bytes(w)
    pf_flops, dec_flops = prefill_flops(p), decode_flops(w)
    decode_gbs = whole_job_rate(dec_b, world, leg_ms["decode"]) / 1e9
    prefill_tflops = whole_job_rate(pf_flops, world, leg_ms["prefill"]) / 1e12
    cw_gbs = whole_job_rate(cw_b, world, leg_ms["cache_write"]) / 1e9
    hbm = float(peaks["hbm_gbs"])
    bf16_burst = float(peaks["bf16_tflops"])
    fp32_alu = SM_COUNT * FP32_LANES * 2 * SM_MAX_MHZ * 1e6 / 1e12  # CUDA-core fp32 FMA peak

    kinds = {k: mla.kernel_kind(k) for k in ("decode", "prefill", "cache_write")}

    def roof(kind, achieved_gbs=None, achieved_tflops=None, kernel=None):
        if kind == "hbm":
            r = {"bound": "hbm", "achieved": achieved_gbs / world, "peak": hbm, "unit": "GB/s"}
        elif kind == "tensor":
            r = {"bound": "tensor", "achieved": achieved_tflops / world, "peak": bf16_burst, "unit": "TFLOP/s"}
        else:
            r = {"bound": "alu", "achieved": achieved_tflops / world, "peak": fp32_alu, "unit": "TFLOP/s"}
        r["frac"] = r["achieved"] / r["peak"]
        r["peak_source"] = f"{peak_src}" if kind != "alu" else "derived: 152 SM x 128 fp32 lanes x 2 x 2070 MHz"
        r["traffic"] = _traffic(kernel) if kernel else None
        return r

    legs_roof = {
        "cache_write": roof("hbm", achieved_gbs=cw_gbs, kernel="cache_write"),
        "decode": roof(kinds["decode"], achieved_gbs=decode_gbs, achieved_tflops=world * dec_flops /
                       (leg_ms["decode"] * 1e-3) / 1e12, kernel="decode"),
        "prefill": roof(kinds["prefill"], achieved_tflops=prefill_tflops, kernel="prefill"),
    }
    dominant = max(leg_ms, key=lambda n: leg_ms[n])

    # --- end to end through the C-ABI call with pinned host buffers -------
    e2e = None
    if args.e2e:
        h_q = w.q.cpu().contiguous().pin_memory()
        h_pt = w.page_table.cpu().contiguous().pin_memory()
        h_sl = w.seq_lens.cpu().pin_memory()
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        d_q, d_pt, d_sl = torch.empty_like(w.q), torch.empty_like(w.page_table), torch.empty_like(w.seq_lens)

        def e2e_decode():
            # one library call: H2D of q / page table / lengths, decode, D2H of out
            mla.mla_nvfp4_decode_host(h_q, d_q, cache, gs, w.softmax_scale, h_out, out,
                                      page_table_host=h_pt, page_table_dev=d_pt, seq_lens_host=h_sl,
                                      seq_lens_dev=d_sl, workspace=ws, error_word=err,
                                      num_splits=decode_splits)

        for _ in range(args.warmup):
            e2e_decode()
        torch.cuda.synchronize()
        times = []
        for _ in range(args.steps):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            e2e_decode()
            e1.record(stream)
            times.append((e0, e1))
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in times) / args.steps
        h2d = h_q.numel() * 2 + h_pt.numel() * 4 + h_sl.numel() * 4
        d2h = h_out.numel() * 2
        e2e = {"value": world * dec_b / (ms * 1e-3) / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms": ms,
               "what": "decode leg through the C-ABI call mla_nvfp4_decode_host: H2D q/page table/lengths "
                       "from pinned memory, decode, D2H of out; cache resident"}

    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item()):#x}")

    line = {
        "metric": METRIC, "value": decode_gbs, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": mla.compute_dtype(), "data": "synthetic (seeded, generated on device)",
        "config": {"workload": WORKLOAD, "parallelism": f"replicas x{world} (independent batches, no collective)",
                   "l2": "flushed by a 256 MB write before every leg", "decode_batch": w.batch,
                   "heads": w.heads, "seq_len": 4096, "record_bytes": w.record_bytes,
                   "prefill_tokens": p.total_tokens},
        "decode": {"ms": leg_ms["decode"], "gbs": decode_gbs, "hbm_frac": decode_gbs / world / hbm,
                   "tflops": world * dec_flops / (leg_ms["decode"] * 1e-3) / 1e12,
                   "bytes": dec_b, "flops": dec_flops},
        "prefill": {"ms": leg_ms["prefill"], "tflops": prefill_tflops,
                    "bf16_frac": prefill_tflops / world / bf16_burst, "flops": pf_flops},
        "cache_write": {"ms": leg_ms["cache_write"], "gbs": cw_gbs, "hbm_frac": cw_gbs / world / hbm,
                        "bytes": cw_b},
        "roofline": dict(legs_roof[dominant], kernel=dominant),
        "roofline_legs": legs_roof,
        "gpu_launches": launches_per_step * args.steps,
        "wall_s_timed_region": wall,
        "e2e": e2e,
        "clocks": clk.summary(),
    }
    return line


# ---------------------------------------------------------------------------
# CPU oracle (test infrastructure): the cpu_baseline leg and --impl reference
# ---------------------------------------------------------------------------
def host_cpu_info():
    """(CPU model, BLAS threads) of the host running the oracle: the oracle's
    heavy steps are NumPy matmuls, so the BLAS pool is the thread count it uses."""
    model = platform.machine()
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.split(":")[0].strip() == "Model name":
                model = f"{ln.split(':', 1)[1].strip()} ({platform.machine()})"
                break
    except (OSError, subprocess.SubprocessError):
        pass
    threads = None
    try:
        from threadpoolctl import threadpool_info
        blas = [i for i in threadpool_info() if i.get("user_api") == "blas"]
        if blas:
            threads = max(int(i["num_threads"]) for i in blas)
    except ImportError:
        pass
    if threads is None:
        for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
            if os.environ.get(var, "").isdigit():
                threads = int(os.environ[var])
                break
    if threads is None:
        threads = len(os.sched_getaffinity(0))  # BLAS default: one thread per available core
    return model, threads


_ORACLE_INPUTS = {}


def _oracle_inputs():
    """The decode batch as the oracle takes it (built once per process; not timed)."""
    if "w" not in _ORACLE_INPUTS:
        import numpy as np
        from mla_attention_nvfp4_gb300 import workloads
        from oracle import attention, nvfp4
        w = workloads.decode_dsv3(device="cpu")
        kv = w.kv_c.float().numpy()
        _ORACLE_INPUTS.update(
            w=w, kv=kv, gs=nvfp4.global_scale(np.abs(kv).max()), pe=w.k_pe.float().numpy(),
            slots=attention.decode_slots_paged(w.page_table.cpu().numpy(), w.seq_lens.cpu().numpy(), 64),
            q=w.q.float().numpy())
    return _ORACLE_INPUTS


def oracle_decode_sample(budget_s: float):
    """Time the float64 oracle on whole sequences of the decode batch until
    the time budget is spent; returns (GB/s in the decode metric, sample)."""
    import numpy as np
    from oracle import attention, cache as ocache

    inp = _oracle_inputs()
    w, kv, gs, pe, slots, q = inp["w"], inp["kv"], inp["gs"], inp["pe"], inp["slots"], inp["q"]
    per_seq = 4096
    t0 = time.perf_counter()
    done = 0
    cache = np.zeros((w.num_slots, w.record_bytes), dtype=np.uint8)
    while done < w.batch and (time.perf_counter() - t0) < budget_s:
        sl = slots[done]
        rows = np.arange(done * per_seq, (done + 1) * per_seq)
        cache[sl] = ocache.encode_records(kv[rows], pe[rows], gs, w.record_bytes)
        attention.decode(q[done:done + 1], cache, w.record_bytes, gs, w.softmax_scale, [sl])
        done += 1
    dt = time.perf_counter() - t0
    rec_bytes = done * per_seq * w.record_bytes + done * w.heads * (576 + 512) * 2 + 64 * 4 + 4
    return rec_bytes / dt / 1e9, f"{done} of {w.batch} decode sequences (cache write + decode, 4096 keys, " \
                                  f"128 heads each) in {dt:.1f} s"


def run_reference(args, rank, world):
    if rank != 0:
        return None
    # each step a bounded sample (at least one whole sequence), the whole run ~90 s
    budget = max(0.25, 90.0 / max(1, args.steps + args.warmup))
    vals = []
    for i in range(args.warmup + args.steps):
        v, sample = oracle_decode_sample(budget)
        if i >= args.warmup:
            vals.append(v)
    value = statistics.mean(vals)
    model, cores = host_cpu_info()
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": WORKLOAD},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
                         "cpu_model": model, "affinity_cores": len(os.sched_getaffinity(0))},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--case", default="full", choices=["full", "profile", "decode-steady"],
                    help="profile: smaller prefill input; decode-steady: decode of 16 x 4096 keys in one "
                         "split (64 tiles per CTA); both for ncu captures, not bench values")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line))
        return

    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    cpu_line = None
    if rank == 0 and world == 1 and args.cpu_baseline:
        # oracle before any CUDA work, so that no forked worker sees a CUDA context
        v, sample = oracle_decode_sample(args.cpu_budget)
        model, cores = host_cpu_info()
        cpu_line = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
                    "cpu_model": model, "affinity_cores": len(os.sched_getaffinity(0))}
    line = run_ours(args, rank, world)
    if args.case != "full":
        what = "prefill 2x4096" if args.case == "profile" else "decode 16x4096, one split"
        line["config"]["workload"] = f"PROFILE CASE ({what}), not a bench value: " + WORKLOAD
    if rank == 0:
        line["cpu_baseline"] = cpu_line
        print(json.dumps(line))
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
