#!/usr/bin/env python
"""Benchmark of the MLA NVFP4 hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input of
every workload the path is specified on:
  1. cache write of the 262,144 latent tokens of the DeepSeek-V3-shaped
     decode batch (64 x 4096) into 432-byte records (bf16 RoPE);
  2. decode of that batch (64 sequences x 128 heads x 4096 keys, 576-d bf16
     queries, random page permutation, length-aware split plan);
  3. causal varlen prefill of 8 x 4096 tokens x 128 heads (q/k 192, v 128)
     with the fused NVFP4 output;
  4. cache write of the mixed-length batch's ~1.17M tokens into 368-byte
     records (fp8 RoPE);
  5. decode of the mixed-length batch (128 sequences, lengths log-uniform
     1k..32k, 128 heads, 368-byte records);
  6. sparse top-k decode (32 queries x 128 heads, 2048 of 65,536 context
     tokens each, a few -1 entries);
  7. the NVFP4 output projection on the prefill's fused output as written
     (32,768 tokens x 16,384 = 128 heads x 128, against a 7168-row NVFP4
     weight), on block-scaled fp4 tensor cores.
Legs are timed with CUDA events on the launching stream; L2 is flushed (a
256 MB write) before every leg.  `value` is the DeepSeek-V3-shaped decode
leg's algorithmic HBM throughput (the metric's first part); every leg's
GB/s, TFLOP/s and roofline fractions are reported beside it.

--impl reference times the CPU oracle (test infrastructure) on a bounded
sample of the decode workload instead.
"""
from __future__ import annotations

import argparse
import datetime
import json
import math
import os
import platform
import socket
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
            "split-K decode, planned from the host-held lengths) + prefill_8x4096: causal varlen H128 qk192 v128 fused NVFP4 out + "
            "decode_mixed: B128 H128 L~logU(1k,32k) 368B fp8-RoPE records (cache write + decode) + "
            "decode_topk: B32 H128 2048 of 65536 tokens, 432B + gemm_oproj: NVFP4 [32768 x 16384] x [7168 x 16384]^T "
            "on the prefill output")
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
SM_COUNT, SM_MAX_MHZ, FP32_LANES = 152, 2070.0, 128
# Dense tensor-core rate of fp4 (block-scaled e2m1) over bf16: 13.5 / 2.25
# PFLOP/s nominal; the fp4 roofline is the measured bf16 peak times this.
FP4_OVER_BF16 = 6.0
CLOCK_SAMPLE_MS = 50


CORE_LEGS = ("cache_write_432", "cache_write_368", "decode_dsv3", "decode_mixed", "decode_topk", "prefill")


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
    """nvidia-smi clock / throttle sampling; summary() keeps the samples
    taken inside the wall-clock window it is given (the timed region)."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
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
                                          "--format=csv,noheader,nounits", "-lms", str(CLOCK_SAMPLE_MS)],
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

    def summary(self, t0=None, t1=None):
        try:
            return summarize_clocks(open(self.path).read().splitlines() if self.proc is not None and
                                    os.path.exists(self.path) else None, t0, t1)
        finally:
            if self.temporary and os.path.exists(self.path):
                os.remove(self.path)


def summarize_clocks(lines, t0=None, t1=None):
    """Median SM clock, max clock and the throttle reasons seen, over the
    nvidia-smi samples whose timestamp lies in [t0, t1] (epoch seconds)."""
    if lines is None:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
    sm, smax, reasons = [], None, set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in lines:
        parts = [x.strip() for x in line.split(",")]
        if len(parts) < 10:
            continue
        try:
            ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            mhz, mx = float(parts[2]), float(parts[3])
        except ValueError:
            continue
        if (t0 is not None and ts < t0) or (t1 is not None and ts > t1):
            continue
        sm.append(mhz)
        smax = mx
        for n, v in zip(names, parts[6:10]):
            if v.lower().startswith("active"):
                reasons.add(n)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": smax, "samples": 0, "reasons": ["unsampled"]}
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "samples": len(sm), "reasons": sorted(reasons)}


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


class CudaTimer:
    """Per-leg CUDA events on the launching stream."""

    def __init__(self, stream):
        import torch
        self.torch, self.stream, self.pairs = torch, stream, []

    def start(self):
        e = self.torch.cuda.Event(enable_timing=True)
        e.record(self.stream)
        return e

    def stop(self, e0):
        e1 = self.torch.cuda.Event(enable_timing=True)
        e1.record(self.stream)
        return (e0, e1)

    def sync(self):
        self.torch.cuda.synchronize()

    @staticmethod
    def ms(mark):
        return mark[0].elapsed_time(mark[1])


class HostTimer:
    """Wall-clock stand-in for CudaTimer (host-only legs, CPU tests)."""

    def start(self):
        return time.perf_counter()

    def stop(self, t0):
        return (t0, time.perf_counter())

    def sync(self):
        pass

    @staticmethod
    def ms(mark):
        return (mark[1] - mark[0]) * 1e3


def time_legs(legs, steps, warmup, timer, before_leg=None, barrier=None):
    """Run `warmup` untimed steps, then `steps` timed ones; a step runs every
    leg once in order, `before_leg` (the L2 flush) before each, outside the
    leg's timing.  Returns (mean ms per leg, wall-clock window (t0, t1) of
    the timed steps)."""
    def step(marks=None):
        for name, fn in legs:
            if before_leg is not None:
                before_leg()
            if marks is None:
                fn()
            else:
                e0 = timer.start()
                fn()
                marks[name].append(timer.stop(e0))

    for _ in range(warmup):
        step()
    timer.sync()
    marks = {name: [] for name, _ in legs}
    if barrier is not None:
        barrier()
    timer.sync()
    t0 = time.time()
    for _ in range(steps):
        step(marks)
    timer.sync()
    t1 = time.time()
    return {n: sum(timer.ms(m) for m in marks[n]) / steps for n in marks}, (t0, t1)


def e2e_pipelined_ms(mla, w, ds, h_q, h_pt, h_sl, err, splits, steps, warmup, dev, barrier=None):
    """Mean ms per step of the host-buffer decode with two steps in flight:
    step i runs on stream i mod 2 with that stream's device buffers, its own
    workspace and cache copy i mod 2 (so consecutive steps read different
    records and no step finds the previous one's in L2), its H2D copies,
    decode and D2H copy all inside the call.  CUDA events: a start event on
    the current stream that both streams wait for, an end event per stream
    that the current stream waits for."""
    import torch
    caches = [ds["cache"], ds["cache"].clone()]
    bufs = []
    for k in range(2):
        need = mla.mla_nvfp4_decode_workspace_size(w.batch, w.heads, splits)
        bufs.append(dict(q=torch.empty_like(w.q), pt=torch.empty_like(w.page_table), sl=torch.empty_like(w.seq_lens),
                         out=torch.empty_like(ds["out"]), h_out=torch.empty(ds["out"].shape, dtype=torch.bfloat16)
                         .pin_memory(), ws=torch.empty(need, dtype=torch.uint8, device=dev) if need > 0 else None,
                         stream=torch.cuda.Stream(device=dev)))

    def step(i):
        b = bufs[i & 1]
        with torch.cuda.stream(b["stream"]):
            mla.mla_nvfp4_decode_host(h_q, b["q"], caches[i & 1], ds["gs"], w.softmax_scale, b["h_out"], b["out"],
                                      page_table_host=h_pt, page_table_dev=b["pt"], seq_lens_host=h_sl,
                                      seq_lens_dev=b["sl"], workspace=b["ws"], error_word=err, num_splits=splits)

    for i in range(max(warmup, 2)):
        step(i)
    torch.cuda.synchronize()
    if barrier is not None:
        barrier()
    cur = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    for b in bufs:
        b["stream"].wait_event(e0)
    for i in range(steps):
        step(i)
    for b in bufs:
        e = torch.cuda.Event()
        e.record(b["stream"])
        cur.wait_event(e)
    e1.record(cur)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def summarize(leg_ms, meta, world, peaks, peak_src, headline="decode_dsv3"):
    """Bench-line fields from per-leg mean times (already max over ranks).
    meta[leg] = {"bytes", "flops", "bound", "dtype", "kernel"}: algorithmic
    bytes and flops of one launch sequence on one rank.  Rates are whole-job
    (weak scaling: world x units over the slowest rank's time); roofline
    fractions are per GPU against the measured peaks."""
    hbm = float(peaks["hbm_gbs"])
    bf16 = float(peaks["bf16_tflops"])
    legs = {}
    for name, ms in leg_ms.items():
        m = meta[name]
        gbs = whole_job_rate(m["bytes"], world, ms) / 1e9
        tflops = whole_job_rate(m["flops"], world, ms) / 1e12 if m["flops"] else None
        leg = {"ms": ms, "gbs": gbs, "hbm_frac": gbs / world / hbm, "dtype": m["dtype"], "bytes": m["bytes"],
               "flops": m["flops"]}
        if tflops is not None:
            leg["tflops"] = tflops
            leg["tensor_frac"] = tflops / world / bf16
        traffic = _traffic(m["kernel"]) if m.get("kernel") else None
        if m["bound"] == "hbm":
            roof = {"bound": "hbm", "achieved": gbs / world, "peak": hbm, "unit": "GB/s"}
            if traffic is not None:
                leg["dram_gbs"] = traffic / (ms * 1e-3) / 1e9
                leg["dram_frac"] = leg["dram_gbs"] / hbm
        else:
            x = m.get("peak_x", 1.0)
            roof = {"bound": "tensor", "achieved": tflops / world, "peak": bf16 * x, "unit": "TFLOP/s"}
            if x != 1.0:
                leg["tensor_frac"] = tflops / world / (bf16 * x)
        roof["frac"] = roof["achieved"] / roof["peak"]
        roof["peak_source"] = peak_src if m.get("peak_x", 1.0) == 1.0 else \
            f"{peak_src} bf16 x {m['peak_x']:g} (nominal fp4 / bf16 dense ratio)"
        roof["traffic"] = traffic
        leg["roofline"] = roof
        legs[name] = leg
    # the dominant kernel of the hot path itself (cache write, decode,
    # prefill, their configs); the extension legs are reported per leg
    core = [n for n in leg_ms if n in CORE_LEGS] or list(leg_ms)
    dominant = max(core, key=lambda n: leg_ms[n])
    return {
        "value": legs[headline]["gbs"],
        "ms_per_step": sum(leg_ms.values()),
        "legs": legs,
        "roofline": dict(legs[dominant]["roofline"], kernel=dominant),
    }


def extension_legs(mla, w, ds, p, gsp, codes, scales, err, dev, step_splits):
    """Legs of the extensions of the hot path, timed in the full case:
    decode with the NVFP4 query, the chunked-context prefill, the
    fake-quantised prefill (dense and 2:4).  Returns (legs, meta, launches
    per step)."""
    import torch
    T, H = p.total_tokens, p.heads
    # decode_dsv3 with the query quantised to NVFP4 (block-scaled fp4 scores)
    gq = mla.mla_nvfp4_global_scale(w.q)

    def leg_q4():
        mla.mla_nvfp4_decode_q4(w.q, ds["cache"], ds["gs"], w.softmax_scale, gq, out=ds["out"], lse=ds["lse"],
                                workspace=ds["ws"], error_word=err, num_splits=step_splits(ds), **ds["kw"])

    # chunked-context prefill: the prefill's tokens after a context of the
    # same length per sequence; the context's latent gathered from the
    # decode cache (one slot per context token), its per-head keys and
    # values (the model's kv_b_proj, a library GEMM left out of the leg)
    # stood in for by tensors of the projected shape
    slots = torch.arange(T, dtype=torch.int64, device=dev) * (ds["w"].num_slots // T)
    kv_g = torch.empty((T, 512), dtype=torch.bfloat16, device=dev)
    pe_g = torch.empty((T, 64), dtype=torch.bfloat16, device=dev)
    o_parts = torch.empty((2, T, H, 128), dtype=torch.float32, device=dev)
    l_parts = torch.empty((2, H, T), dtype=torch.float32, device=dev)

    def leg_chunked():
        mla.mla_nvfp4_gather_latent(ds["cache"], ds["gs"], slots, kv_c=kv_g, k_pe=pe_g, error_word=err)
        mla.mla_nvfp4_prefill_partial(p.q, p.k, p.v, p.cu_seqlens, p.max_seqlen, p.softmax_scale,
                                      cu_seqlens_k=p.cu_seqlens, out=o_parts[0], lse=l_parts[0], error_word=err)
        mla.mla_nvfp4_prefill_partial(p.q, p.k, p.v, p.cu_seqlens, p.max_seqlen, p.softmax_scale,
                                      out=o_parts[1], lse=l_parts[1], error_word=err)
        mla.mla_nvfp4_merge_fused_out(o_parts, l_parts, gsp, out_codes=codes, out_scales=scales, error_word=err)

    # fake-quantised prefill: operand quantisation pass plus the attention
    gs3 = [mla.mla_nvfp4_global_scale(t) for t in (p.q, p.k, p.v)]
    qc = mla.mla_nvfp4_prefill_qdq(p.q, p.k, p.v, p.cu_seqlens, p.max_seqlen, *gs3, error_word=err)

    def fq(sparse):
        def leg():
            mla.mla_nvfp4_prefill_qdq(p.q, p.k, p.v, p.cu_seqlens, p.max_seqlen, *gs3, error_word=err)
            mla.mla_nvfp4_prefill_fakequant(*qc, p.cu_seqlens, p.max_seqlen, p.softmax_scale, *gs3, gsp,
                                            sparse24=sparse, out_codes=codes, out_scales=scales, error_word=err)
        return leg

    lens = (p.cu_seqlens[1:] - p.cu_seqlens[:-1]).to("cpu", torch.int64)
    ctx_flops = 2.0 * int((lens * lens).sum()) * H * (192 + 128)
    qkv_bytes = T * H * (192 * 2 + 128) * 2
    meta = {
        "decode_dsv3_q4": dict(bytes=decode_bytes(w), flops=decode_flops(w), bound=mla.kernel_kind("decode"),
                               dtype="nvfp4 scores, f16 P.V", kernel=None),
        "prefill_chunked": dict(bytes=prefill_bytes(p) + qkv_bytes + T * (432 + 512 * 2 + 64 * 2 + 8)
                                + 2 * 2 * T * H * 128 * 4, flops=prefill_flops(p) + ctx_flops,
                                bound="tensor", dtype="bf16", kernel=None),
        "prefill_fakequant": dict(bytes=prefill_bytes(p) + 2 * qkv_bytes, flops=prefill_flops(p), bound="tensor",
                                  dtype="f16 (NVFP4 code*scale operands)", kernel=None),
        "prefill_fakequant_24": dict(bytes=prefill_bytes(p) + 2 * qkv_bytes, flops=prefill_flops(p), bound="tensor",
                                     dtype="f16 (NVFP4 code*scale operands)", kernel=None),
    }
    legs = [("decode_dsv3_q4", leg_q4), ("prefill_chunked", leg_chunked), ("prefill_fakequant", fq(False)),
            ("prefill_fakequant_24", fq(True))]
    L = mla.LAUNCHES_PER_CALL
    launches = mla.decode_launches(w.batch, w.heads, ds["splits_used"]) + L["gather_latent"] + 2 * L["prefill_partial"] + \
        L["merge_fused_out"] + 2 * (L["prefill_qdq"] + L["prefill_fakequant"])
    return legs, meta, launches


def run_ours(args, rank, world):
    import torch
    import mla_attention_nvfp4_gb300 as mla
    from mla_attention_nvfp4_gb300 import workloads

    torch.cuda.set_device(rank % max(1, torch.cuda.device_count()))
    dev = torch.device("cuda", torch.cuda.current_device())
    mla.load_library()
    peaks, peak_src = _peaks()
    stream = torch.cuda.current_stream()
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    # --- workloads (device-resident), seed 0 ----------------------------
    steady = args.case == "decode-steady"
    w = workloads.decode_dsv3(device=dev, batch=16 if steady else 64)
    decode_splits = 1 if steady else 0
    if args.case == "profile":
        # the same legs on a prefill of 2 x 4096 tokens (about 1.8 GB on the
        # device in all), for ncu captures; never a bench value
        p = workloads.prefill("prefill_2x4096", seq_lens=(4096, 4096), device=dev)
    else:
        p = workloads.prefill_8x4096(device=dev)
    full = args.case == "full"
    wm = workloads.decode_mixed(device=dev) if full else None
    wt = workloads.decode_topk(device=dev) if full else None

    def decode_setup(wl, splits):
        gs = mla.mla_nvfp4_global_scale(wl.kv_c)
        cache = torch.zeros((wl.num_slots, wl.record_bytes), dtype=torch.uint8, device=dev)
        out = torch.empty((wl.batch, wl.heads, 512), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((wl.batch, wl.heads), dtype=torch.float32, device=dev)
        need = mla.mla_nvfp4_decode_workspace_size(wl.batch, wl.heads, splits)
        ws = torch.empty(need, dtype=torch.uint8, device=dev) if need > 0 else None
        kw = dict(page_table=wl.page_table, seq_lens=wl.seq_lens) if wl.paged else \
            dict(topk_indices=wl.topk_indices)
        d = dict(w=wl, gs=gs, cache=cache, out=out, lse=lse, ws=ws, kw=kw, splits=splits,
                 lens_host=wl.seq_lens.cpu() if wl.paged else None)
        d["splits_used"] = step_splits(d)
        return d

    def step_splits(d):
        # paged calls left to the plan: the lengths are also held on the host
        # (a serving scheduler has them there), so the plan's choice is made
        # there each step; one chunk per sequence runs as the one-split launch
        if d["splits"] == 0 and d["lens_host"] is not None and d["ws"] is not None:
            return mla.mla_nvfp4_decode_plan_splits(d["lens_host"], d["w"].heads, d["ws"].numel())
        return d["splits"]

    def cache_write(d):
        wl = d["w"]
        return lambda: mla.mla_nvfp4_cache_write(wl.kv_c, wl.k_pe, wl.slot_mapping, d["cache"], d["gs"], err)

    def decode(d):
        wl = d["w"]
        return lambda: mla.mla_nvfp4_decode(wl.q, d["cache"], d["gs"], wl.softmax_scale, out=d["out"], lse=d["lse"],
                                            workspace=d["ws"], error_word=err, num_splits=step_splits(d), **d["kw"])

    ds = decode_setup(w, decode_splits)
    gsp = mla.mla_nvfp4_global_scale(p.v)
    codes = torch.empty((p.total_tokens, p.heads * 64), dtype=torch.uint8, device=dev)
    scales = torch.empty(mla.prefill_scale_bytes(p.total_tokens, p.heads), dtype=torch.uint8, device=dev)

    def leg_prefill():
        mla.mla_nvfp4_prefill_fused_out(p.q, p.k, p.v, p.cu_seqlens, p.max_seqlen, p.softmax_scale, gsp,
                                        out_codes=codes, out_scales=scales, error_word=err)

    legs = [("cache_write_432", cache_write(ds)), ("decode_dsv3", decode(ds)), ("prefill", leg_prefill)]
    # output projection weight: random NVFP4 [7168, H*128] (codes and
    # scales in a moderate range), and the GEMM's bf16 output
    n_out, k_in = 7168, p.heads * 128
    gw = torch.Generator(device=dev)
    gw.manual_seed(7)
    w_codes = torch.randint(0, 256, (n_out, k_in // 2), dtype=torch.uint8, device=dev, generator=gw)
    w_sf = torch.randint(0x28, 0x48, (n_out * k_in // 16,), dtype=torch.uint8, device=dev, generator=gw)
    gs_w = torch.tensor([1.0 / 4096], device=dev)
    o_proj = torch.empty((p.total_tokens, n_out), dtype=torch.bfloat16, device=dev)

    def leg_gemm():
        mla.mla_nvfp4_gemm(codes, scales, w_codes, w_sf, gsp, gs_w, out=o_proj)

    with_gemm = args.case != "decode-steady"
    if with_gemm:
        legs.append(("gemm_oproj", leg_gemm))
    meta = {
        "cache_write_432": dict(bytes=cache_write_bytes(w), flops=0, bound="hbm", dtype="fp32->nvfp4",
                                kernel="cache_write"),
        "decode_dsv3": dict(bytes=decode_bytes(w), flops=decode_flops(w), bound=mla.kernel_kind("decode"),
                            dtype=mla.operand_dtype("decode"), kernel="decode"),
        "prefill": dict(bytes=prefill_bytes(p), flops=prefill_flops(p), bound=mla.kernel_kind("prefill"),
                        dtype=mla.operand_dtype("prefill"), kernel="prefill"),
        "gemm_oproj": dict(bytes=p.total_tokens * k_in // 2 + n_out * k_in // 2 + (p.total_tokens + n_out) * k_in // 16
                           + p.total_tokens * n_out * 2, flops=2.0 * p.total_tokens * n_out * k_in,
                           bound=mla.kernel_kind("gemm"), dtype=mla.operand_dtype("gemm"), kernel=None,
                           peak_x=FP4_OVER_BF16),
    }
    launches = mla.LAUNCHES_PER_CALL["cache_write"] + mla.decode_launches(w.batch, w.heads, ds["splits_used"]) + \
        mla.LAUNCHES_PER_CALL["prefill"] + (mla.LAUNCHES_PER_CALL["gemm"] if with_gemm else 0)
    if full:
        dm, dt = decode_setup(wm, 0), decode_setup(wt, 0)
        cache_write(dt)()  # the top-k cache is written once, outside the timed legs
        legs += [("cache_write_368", cache_write(dm)), ("decode_mixed", decode(dm)), ("decode_topk", decode(dt))]
        meta.update({
            # the committed traffic figure is for the 432-byte launch only
            "cache_write_368": dict(bytes=cache_write_bytes(wm), flops=0, bound="hbm", dtype="fp32->nvfp4",
                                    kernel=None),
            "decode_mixed": dict(bytes=decode_bytes(wm), flops=decode_flops(wm), bound=mla.kernel_kind("decode"),
                                 dtype=mla.operand_dtype("decode"), kernel=None),
            "decode_topk": dict(bytes=decode_bytes(wt), flops=decode_flops(wt), bound=mla.kernel_kind("decode"),
                                dtype=mla.operand_dtype("decode"), kernel=None),
        })
        launches += mla.LAUNCHES_PER_CALL["cache_write"] + mla.decode_launches(wm.batch, wm.heads, dm["splits_used"]) + \
            mla.decode_launches(wt.batch, wt.heads, 0, paged=False)
        legs_next, meta_next, launches_next = extension_legs(mla, w, ds, p, gsp, codes, scales, err, dev, step_splits)
        legs += legs_next
        meta.update(meta_next)
        launches += launches_next
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    barrier = (lambda: torch.distributed.barrier()) if world > 1 else None
    with ClockSampler(dev.index) as clk:
        leg_ms, (t0, t1) = time_legs(legs, args.steps, args.warmup, CudaTimer(stream),
                                     before_leg=flush.zero_, barrier=barrier)
        torch.cuda.synchronize()
        if int(err.item()) != 0:
            raise RuntimeError(f"device error word {int(err.item()):#x}")
    clocks = clk.summary(t0, t1)
    names = list(leg_ms)
    leg_ms = dict(zip(names, max_over_ranks([leg_ms[n] for n in names], world, dev)))
    line = summarize(leg_ms, meta, world, peaks, peak_src)

    # --- end to end through the C-ABI call with pinned host buffers -------
    e2e = None
    if args.e2e:
        h_q = w.q.cpu().contiguous().pin_memory()
        h_pt = w.page_table.cpu().contiguous().pin_memory()
        h_sl = w.seq_lens.cpu().pin_memory()
        h_out = torch.empty(ds["out"].shape, dtype=torch.bfloat16).pin_memory()
        d_q, d_pt, d_sl = torch.empty_like(w.q), torch.empty_like(w.page_table), torch.empty_like(w.seq_lens)

        def e2e_decode():
            # one library call: H2D of q / page table / lengths, decode, D2H of out
            mla.mla_nvfp4_decode_host(h_q, d_q, ds["cache"], ds["gs"], w.softmax_scale, h_out, ds["out"],
                                      page_table_host=h_pt, page_table_dev=d_pt, seq_lens_host=h_sl,
                                      seq_lens_dev=d_sl, workspace=ds["ws"], error_word=err,
                                      num_splits=decode_splits)

        e2e_ms, _ = time_legs([("e2e", e2e_decode)], args.steps, args.warmup, CudaTimer(stream),
                              before_leg=flush.zero_, barrier=barrier)
        serial_ms = max_over_ranks([e2e_ms["e2e"]], world, dev)[0]
        ms = max_over_ranks([e2e_pipelined_ms(mla, w, ds, h_q, h_pt, h_sl, err, decode_splits, args.steps,
                                              args.warmup, dev, barrier)], world, dev)[0]
        h2d = h_q.numel() * 2 + h_pt.numel() * 4 + h_sl.numel() * 4
        d2h = h_out.numel() * 2
        e2e = {"value": whole_job_rate(decode_bytes(w), world, ms) / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms": ms, "serial_ms": serial_ms,
               "serial_value": whole_job_rate(decode_bytes(w), world, serial_ms) / 1e9,
               "what": "decode_dsv3 leg through the C-ABI call mla_nvfp4_decode_host, one call per step: H2D of "
                       "q/page table/lengths from pinned memory, decode, D2H of out.  value/ms: two steps in "
                       "flight on two streams (each with its own device buffers and workspace), so one step's "
                       "copies overlap the other's decode; the steps alternate between two copies of the cache "
                       "(226 MB read per two steps, more than L2); time of all steps / steps.  serial_value/"
                       "serial_ms: one step at a time on one stream, L2 flushed before each"}

    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item()):#x}")

    out = {
        "metric": METRIC, "value": line["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": line["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": mla.operand_dtype("decode"),
        "data": "synthetic (seeded, generated on device)",
        "config": {"workload": WORKLOAD, "parallelism": f"replicas x{world} (independent batches, no collective)",
                   "l2": "flushed by a 256 MB write before every leg", "decode_batch": w.batch,
                   "heads": w.heads, "seq_len": 4096, "record_bytes": w.record_bytes,
                   "prefill_tokens": p.total_tokens},
        "legs": line["legs"],
        "roofline": line["roofline"],
        "gpu_launches": launches * args.steps,
        "wall_s_timed_region": t1 - t0,
        "e2e": e2e,
        "clocks": clocks,
    }
    # the former top-level leg keys, kept for readers of earlier lines
    out["decode"] = line["legs"]["decode_dsv3"]
    out["prefill"] = line["legs"]["prefill"]
    out["cache_write"] = line["legs"]["cache_write_432"]
    return out


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


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def launch_ranks(n: int, argv) -> int:
    """Run this script as n ranks (one process per GPU) through
    torch.distributed.run on 127.0.0.1; returns their exit status."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", os.path.abspath(__file__)] + list(argv)
    return subprocess.call(cmd)


def main(argv=None):
    argv = sys.argv[1:] if argv is None else argv
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--case", default="full", choices=["full", "profile", "decode-steady"],
                    help="profile: smaller prefill input; decode-steady: decode of 16 x 4096 keys in one "
                         "split (64 tiles per CTA); both without the mixed-length and top-k legs, for ncu "
                         "captures, not bench values")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")

    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # not started by a launcher: start one rank per GPU ourselves
        return launch_ranks(args.gpus, argv)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}", file=sys.stderr)
        return 2
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line))
        return 0

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
    return 0


if __name__ == "__main__":
    sys.exit(main())
