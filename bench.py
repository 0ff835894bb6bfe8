#!/usr/bin/env python3
"""Benchmark of the fused MXFP4 MoE forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step = one moe_mxfp4_forward call (route -> quant -> stage-1 GEMM ->
stage-2 GEMM with the top-k sum) over one batch of synthetic inputs already
resident in HBM.  The default workload is the largest one-GPU configuration,
the skewed prefill batch (T=4096, d_model 7168, d_inter 256, E 257, topk 9).
Between steps the L2 is flushed (a 256 MiB write), so every step reads the
expert weights from HBM.  Step time is the device time between CUDA events the
library records on its stream before its first and after its last kernel.

Multi-GPU (torchrun, one process per GPU): replicas only -- each rank runs an
independent forward on its own batch (the op has no exchange step); the value
is the tokens of all ranks divided by the slowest rank's time (weak scaling).

--impl reference times the CPU oracle (test infrastructure, plain C) on a
bounded sample of the same workload; under torchrun only rank 0 runs it.

Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused MoE µs/call and tokens/s; achieved HBM TB/s or MXFP4 TFLOPS vs roofline"
DEFAULT_WORKLOAD = "prefill_zipf_T4096_D7168_I256_E257_K9"
# Published number for this workload on the pages (MI355X, aiter): 152.7 us/call
# for (T=16, E=257, d_inter=256, topk=9); context only.
PUBLISHED_US = {"decode_T16_D7168_I256_E257_K9": 152.7,
                "decode_T128_D7168_I256_E257_K9": 239.0,
                "dense_T512_D7168_I2048_E33_K9": 380.4}
HBM_FALLBACK_GBS = 6800.0
BF16_FALLBACK_TFLOPS = 1900.0
# nominal dense fp4 : bf16 tensor rate of the part (13.5 : 2.25 PFLOP/s)
FP4_OVER_BF16 = 6.0
L2_FLUSH_BYTES = 256 << 20
KERNEL_SOURCES = [os.path.join(ROOT, "mixture_experts_mxfp4_gb300", "csrc", f)
                  for f in ("gemm.cu", "ptx.cuh", "mx.cuh", "moe_internal.h", "api.cu")]


def profile_summary(workload: str) -> str:
    """Committed ncu summary of the GEMM kernel on this workload."""
    return os.path.join(ROOT, "profiles", f"gemm_{workload}.md")


# ---------------------------------------------------------------- helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Maximum of a per-rank float over all ranks (identity when world == 1)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput: units processed by all ranks / slowest rank's time."""
    return units_per_rank * world / max_seconds


def measured_peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, kind) from MEASURED_PEAKS.json, else the
    recipe's fallback figures."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", BF16_FALLBACK_TFLOPS)), "measured"
    except Exception:
        return HBM_FALLBACK_GBS, BF16_FALLBACK_TFLOPS, "fallback"


def _code_only(text: str) -> str:
    """C/C++/CUDA source without its comments and blank space, so that editing a
    comment does not mark a profile of the same code as stale."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash() -> str:
    """Hash of the code (comments and spacing excluded) of the sources the GEMM
    kernel and its launch geometry are built from; profile summaries record it."""
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per GEMM-kernel launch from the committed ncu summary, or None when
    the summary is missing or the kernel sources changed since it was taken."""
    try:
        text = open(profile_summary(workload)).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_code_sha256_16:\s*([0-9a-f]+)", text)
    m_tr = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if not m_hash or not m_tr or m_hash.group(1) != kernel_source_hash():
        return None
    return int(m_tr.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def alg_flops(w, ids):
    """Algorithmic operations of one call: 6 * (valid routes) * d_model * d_inter
    (stage 1: 2*2I*D per route, stage 2: 2*D*I per route; padding excluded)."""
    import numpy as np

    ids = np.asarray(ids).reshape(-1)
    r_valid = int(((ids >= 0) & (ids < w.E)).sum())
    return 6.0 * r_valid * w.D * w.I


def tensor_peak(moe, stream, dev):
    """Measured dense MXFP4 rate (TFLOP/s) of the library's tensor-core probe: one
    CTA per SM issuing back-to-back M=128 N=256 K=64 mxf4 MMAs for ~20 ms, timed
    with events on the launching stream (best of 3), plus the rate with one
    scale-factor copy per MMA and at the decode kernels' MMA width N=16."""
    import torch

    def run(n, iters, copies, variant=0):
        best = 0.0
        for _ in range(3):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fl = moe.tensor_probe(n, iters, copies, variant, stream.cuda_stream)
            e1.record(stream)
            e1.synchronize()
            best = max(best, fl / (e0.elapsed_time(e1) * 1e-3) / 1e12)
        return best

    run(256, 2000, 0)  # warm-up
    out = {"n256": run(256, 200000, 0), "n256_copy1": run(256, 100000, 1),
           "n128": run(128, 200000, 0), "n16": run(16, 200000, 0), "n16_copy1": run(16, 100000, 1),
           # copy shape and issuing warp (variant bits: 128x256b copies; a second warp)
           "n16_copy1_wide": run(16, 100000, 1, 1), "n16_copy1_warp2": run(16, 100000, 1, 2),
           "n256_copy1_warp2": run(256, 100000, 1, 2)}
    torch.cuda.synchronize(dev)
    return out


def alg_bytes(w, ids, bf16_act=False):
    """Algorithmic bytes of one forward call and of its GEMM kernel (both stages:
    the touched experts' weights and scales, and the quantised hidden rows, or
    the bf16 ones for the bf16-activation forward)."""
    import workloads

    E_t = workloads.touched_experts(ids, w.E)
    per_expert_w13 = 2 * w.I * w.D * 17 // 32      # w13 + its e8m0 scales
    per_expert_w2 = w.D * w.I * 17 // 32           # w2 + scales
    act = w.T * w.D * 2                            # bf16 hidden in
    out = w.T * w.D * 2                            # bf16 out
    route = w.T * w.K * 8                          # ids + weights
    total = E_t * (per_expert_w13 + per_expert_w2) + act + out + route
    gemm = E_t * (per_expert_w13 + per_expert_w2) + (w.T * w.D * 2 if bf16_act else w.T * w.D * 17 // 32)
    return total, gemm, E_t


# ---------------------------------------------------------------- reference arm

def run_reference(args, w):
    """Time the CPU oracle (as it stands) on a bounded sample of the workload."""
    import numpy as np

    import oracle
    import workloads

    inp = workloads.to_numpy(workloads.make_inputs(w))
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    # A step is the oracle on a sample of the batch's tokens (routing over the whole
    # batch), sized from one untimed probe call so that the W warm-up and K timed
    # steps take about --ref-budget-s seconds (at most --ref-tokens tokens a step).
    nmax = min(w.T, max(1, args.ref_tokens))
    t0 = time.perf_counter()
    oracle.forward(**inp, tokens=np.arange(nmax, dtype=np.int32), threads=threads, want_h=False)
    per_tok = (time.perf_counter() - t0) / nmax
    calls = max(1, args.steps) + max(0, args.warmup)
    ntok = int(min(nmax, max(1, args.ref_budget_s / (calls * per_tok))))
    toks = np.arange(ntok, dtype=np.int32)
    for _ in range(max(0, args.warmup)):
        oracle.forward(**inp, tokens=toks, threads=threads, want_h=False)
    times = []
    for _ in range(max(1, args.steps)):
        t0 = time.perf_counter()
        oracle.forward(**inp, tokens=toks, threads=threads, want_h=False)
        times.append(time.perf_counter() - t0)
    tot = sum(times)
    value = ntok * len(times) / tot
    return {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1, "steps": len(times),
        "warmup": args.warmup, "ms_per_step": 1e3 * tot / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": w.name, "T": w.T, "d_model": w.D, "d_inter": w.I, "E": w.E,
                   "topk": w.K, "sample_tokens": ntok},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"{ntok} of {w.T} tokens per step (sized for a "
                                   f"{args.ref_budget_s:g} s run), routing over the whole batch"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def cpu_baseline(w, budget_s: float):
    """Oracle on the host cores over a bounded sample of the workload: whole batches
    while one takes under budget_s, else the batch's first n tokens (routing over
    the whole batch) with n sized from a probe call to take about budget_s."""
    import numpy as np

    import oracle
    import workloads

    inp = workloads.to_numpy(workloads.make_inputs(w))
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    nprobe = min(w.T, 16)
    t0 = time.perf_counter()
    oracle.forward(**inp, tokens=np.arange(nprobe, dtype=np.int32), threads=threads, want_h=False)
    per_tok = (time.perf_counter() - t0) / nprobe
    if per_tok * w.T <= budget_s:
        t0 = time.perf_counter()
        reps = 0
        while True:
            oracle.forward(**inp, threads=threads, want_h=False)
            reps += 1
            if time.perf_counter() - t0 > budget_s:
                break
        dt = time.perf_counter() - t0
        return {"value": w.T * reps / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                "sample": f"{reps} full batches of {w.T} tokens ({w.name}), {dt:.1f} s"}
    ntok = int(max(1, min(w.T, budget_s / per_tok)))
    t0 = time.perf_counter()
    oracle.forward(**inp, tokens=np.arange(ntok, dtype=np.int32), threads=threads, want_h=False)
    dt = time.perf_counter() - t0
    return {"value": ntok / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"the first {ntok} of {w.T} tokens of one batch ({w.name}; routing over "
                      f"the whole batch), {dt:.1f} s"}


# ---------------------------------------------------------------- GPU arm

def run_gpu(args, w, world, rank, local):
    import numpy as np
    import torch

    import mixture_experts_mxfp4_gb300 as moe
    import workloads

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    moe.load_library()
    inp = workloads.make_inputs(w, seed=args.seed + rank)
    t = {k: v.to(dev) for k, v in inp.items()}
    bf16_act = args.activations == "bf16"
    m = moe.MoeMXFP4(w.T, w.D, w.I, w.E, w.K, device=dev,
                     activations="bf16" if bf16_act else "mxfp4")
    out = torch.empty(w.T, w.D, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    fargs = (t["hidden"], t["w13"], t["w13_scale"], t["w2"], t["w2_scale"], t["topk_ids"],
             t["topk_weights"])

    # launch mode: the library's automatic choice unless forced
    moe.set_single_launch({"auto": 2, "single": 1, "separate": 0}[args.launch])
    # (the bf16-activation forward: separate kernels, a separate top-k sum; routing in
    # three launches from 4096 routes)
    launches = ((6 if w.T * w.K >= 4096 else 4) if bf16_act
                else moe.call_launches(w.T, w.D, w.I, w.E, w.K))
    # single launch: the GEMM kernel (routing and quantisation inside) and the top-k sum
    single = launches == 2 and not bf16_act
    moe.set_kernel_timing(2)
    for _ in range(args.warmup):
        flush.zero_()
        m.forward(*fargs, out=out)
    torch.cuda.synchronize(dev)
    if m.device_status() != 0:
        raise RuntimeError("device status after warm-up")

    # Timed region 1 (the headline): events only around each whole call, so the
    # kernels overlap their launches as in normal use.
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.2)  # let the sampler start before the timed region
    total_ms = 0.0
    for _ in range(args.steps):
        flush.zero_()
        m.forward(*fargs, out=out)
        total_ms += moe.last_call_ms()
    torch.cuda.synchronize(dev)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()

    # The same calls without the L2 flush in between (the pages' own timing loop
    # does not flush); reported beside the headline, which is flushed.
    warm_ms = 0.0
    warm_steps = max(1, min(args.steps, 500))
    for _ in range(warm_steps):
        m.forward(*fargs, out=out)
        warm_ms += moe.last_call_ms()
    torch.cuda.synchronize(dev)
    warm_us = 1e3 * warm_ms / warm_steps

    # Timed region 2: events around every kernel (serialises them) for the
    # per-kernel breakdown and the dominant kernel's roofline.
    moe.set_kernel_timing(1)
    names = moe.KERNEL_NAMES
    per_kernel = {n: 0.0 for n in names}
    k_steps = max(1, min(args.steps, 500))
    for _ in range(k_steps):
        flush.zero_()
        m.forward(*fargs, out=out)
        kt = moe.kernel_times()
        for n in names:
            per_kernel[n] = None if kt[n] is None else per_kernel[n] + kt[n]
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if m.device_status() != 0:
        raise RuntimeError("device status after timed region")
    moe.set_kernel_timing(0)

    max_s = max_over_ranks(total_ms / 1e3, world, dev if world > 1 else None)
    value = aggregate_value(w.T * args.steps, world, max_s)
    us_call = 1e3 * total_ms / args.steps

    # ---- end to end through the public API: pinned host in, host out.  The step's
    # inputs (hidden rows, expert ids, weights) sit in one pinned buffer and go over
    # in one copy; the forward takes device pointers into it.
    hb = inp["hidden"].numel() * 2
    ib = inp["topk_ids"].numel() * 4
    wb = inp["topk_weights"].numel() * 4
    h_pack = torch.empty(hb + ib + wb, dtype=torch.uint8).pin_memory()
    h_pack[:hb].copy_(inp["hidden"].contiguous().view(torch.uint8).reshape(-1))
    h_pack[hb:hb + ib].copy_(inp["topk_ids"].contiguous().view(torch.uint8).reshape(-1))
    h_pack[hb + ib:].copy_(inp["topk_weights"].contiguous().view(torch.uint8).reshape(-1))
    h_out = torch.empty(w.T, w.D, dtype=torch.bfloat16).pin_memory()
    d_pack = torch.empty(hb + ib + wb, dtype=torch.uint8, device=dev)
    d_hidden = d_pack[:hb].view(torch.bfloat16).view(w.T, w.D)
    d_ids = d_pack[hb:hb + ib].view(torch.int32).view(w.T, w.K)
    d_w = d_pack[hb + ib:].view(torch.float32).view(w.T, w.K)
    e2e_steps = max(1, min(args.steps, 200))
    for _ in range(3):
        d_pack.copy_(h_pack, non_blocking=True)
        m.forward(d_hidden, *fargs[1:5], d_ids, d_w, out=out)
        h_out.copy_(out, non_blocking=True)
    torch.cuda.synchronize(dev)
    e2e_ms = 0.0
    for _ in range(e2e_steps):
        flush.zero_()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        d_pack.copy_(h_pack, non_blocking=True)
        m.forward(d_hidden, *fargs[1:5], d_ids, d_w, out=out)
        h_out.copy_(out, non_blocking=True)
        s1.record(stream)
        s1.synchronize()
        e2e_ms += s0.elapsed_time(s1)
    # ---- the same call with host buffers passed straight to the API: the kernels
    # read the step's pinned inputs and write its pinned output in place (mapped
    # host memory; NVLink-C2C on GB300), so the transfers are part of the kernels
    # and no staging copy runs.  This is the end-to-end number reported as e2e.
    hh = h_pack[:hb].view(torch.bfloat16).view(w.T, w.D)
    hi = h_pack[hb:hb + ib].view(torch.int32).view(w.T, w.K)
    hw = h_pack[hb + ib:].view(torch.float32).view(w.T, w.K)
    h_out2 = torch.empty(w.T, w.D, dtype=torch.bfloat16).pin_memory()
    e2e_host_ms = None
    try:
        for _ in range(3):
            m.forward(hh, *fargs[1:5], hi, hw, out=h_out2)
        torch.cuda.synchronize(dev)
        e2e_host_ms = 0.0
        for _ in range(e2e_steps):
            flush.zero_()
            s0 = torch.cuda.Event(enable_timing=True)
            s1 = torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            m.forward(hh, *fargs[1:5], hi, hw, out=h_out2)
            s1.record(stream)
            s1.synchronize()
            e2e_host_ms += s0.elapsed_time(s1)
    except ValueError as exc:  # pinned memory the device cannot address in place
        print(f"host-buffer calls not measured: {exc}", file=sys.stderr)
        e2e_host_ms = None
    if e2e_host_ms is not None:
        if m.device_status() != 0:
            raise RuntimeError("device status after the host-buffer calls")
        if not torch.equal(h_out2.view(torch.int16), h_out.view(torch.int16)):
            raise RuntimeError("host-buffer call differs from the device-buffer call")
    # ---- the same call captured in a CUDA graph and replayed (L2 flushed between
    # replays, events around each replay); reported beside the direct calls
    graph_us = None
    try:
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            m.forward(*fargs, out=out)
        stream.wait_stream(cap)
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            m.forward(*fargs, out=out)
        g_ms = 0.0
        g_steps = max(1, min(args.steps, 200))
        for _ in range(g_steps + 3):
            flush.zero_()
            g0 = torch.cuda.Event(enable_timing=True)
            g1 = torch.cuda.Event(enable_timing=True)
            g0.record(stream)
            graph.replay()
            g1.record(stream)
            g1.synchronize()
            g_ms += g0.elapsed_time(g1) if _ >= 3 else 0.0
        if m.device_status() != 0:
            raise RuntimeError("device status after graph replays")
        graph_us = 1e3 * g_ms / g_steps
    except Exception as exc:  # reported, not fatal: the direct calls are the metric
        print(f"graph replay not measured: {exc}", file=sys.stderr)
    e2e_max = max_over_ranks(e2e_ms / 1e3, world, dev if world > 1 else None)
    e2e_staged = aggregate_value(w.T * e2e_steps, world, e2e_max)
    in_place = e2e_host_ms is not None
    if not in_place:  # report the staged path as the end-to-end number
        e2e_host_ms = e2e_ms
    e2e_host_max = max_over_ranks(e2e_host_ms / 1e3, world, dev if world > 1 else None)
    e2e_value = aggregate_value(w.T * e2e_steps, world, e2e_host_max)
    h2d = h_pack.numel()
    d2h = h_out.numel() * 2

    # ---- roofline of the dominant kernel (the GEMM kernel), measured live above
    ids_np = inp["topk_ids"].numpy()
    b_total, b_gemm, e_touched = alg_bytes(w, ids_np, bf16_act)
    flops = alg_flops(w, ids_np)
    peak, bf16_peak, peak_kind = measured_peaks()
    probe = tensor_peak(moe, stream, dev)
    mxf4_peak = probe["n256"]
    ran = {n: v for n, v in per_kernel.items() if v is not None}
    dom = max(ran, key=ran.get)
    g_ms = per_kernel["gemm"] / k_steps
    achieved = b_gemm / (g_ms * 1e-3) / 1e9
    g_tflops = flops / (g_ms * 1e-3) / 1e12
    t_hbm = b_gemm / (peak * 1e9)
    t_fp4 = flops / (mxf4_peak * 1e12)
    roofline = {"bound": "hbm" if t_hbm >= t_fp4 else "tensor", "kernel": "gemm",
                "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                # the committed ncu summary of this workload's GEMM kernel (default launch
                # mode), null once the kernel sources have changed since it was taken
                "traffic": profiled_traffic(w.name) if (not bf16_act and args.launch == "auto")
                else None,
                "alg_bytes_per_launch": b_gemm, "peak_kind": peak_kind,
                "flops_alg": flops, "achieved_tflops": g_tflops,
                "tensor_peak_tflops": mxf4_peak,
                "tensor_peak_kind": "measured: the library's mxf4 probe (M128 N256 K64 MMAs, one CTA "
                                    "per SM, operands in shared memory)",
                "tensor_frac": g_tflops / mxf4_peak,
                "tensor_peak_from_bf16_tflops": bf16_peak * FP4_OVER_BF16,
                "tensor_frac_vs_bf16_ratio": g_tflops / (bf16_peak * FP4_OVER_BF16),
                "t_hbm_us": t_hbm * 1e6, "t_fp4_us": t_fp4 * 1e6,
                "probe_tflops": probe}
    fwd_gbs = b_total / (us_call * 1e-6) / 1e9
    res = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 x bf16 (e2m1 weights expanded in shared memory), fp32 accumulate" if bf16_act
        else "mxfp4 (e2m1 x e2m1, fp32 accumulate)",
        "data": "synthetic (seeded; DeepSeek-R1-shaped, random weights)",
        "config": {"workload": w.name, "T": w.T, "d_model": w.D, "d_inter": w.I, "E": w.E,
                   "topk": w.K, "touched_experts": e_touched,
                   "l2": "flushed before every step (256 MiB write, untimed)",
                   "parallelism": f"replicas x{world}",
                   "activations": "bf16 (W4A16: weights dequantised to bf16 in shared memory)"
                   if bf16_act else "mxfp4 (quantised per 32 elements)",
                   "launch": "single (routing + quantisation inside the GEMM kernel)"
                   if single else "separate kernels"},
        "us_per_call": us_call,
        "us_per_call_graph_replay": graph_us,
        "us_per_call_l2_not_flushed": warm_us,
        "per_kernel_us": {n: (None if v is None else 1e3 * v / k_steps) for n, v in per_kernel.items()},
        "per_kernel_note": f"{k_steps} steps with events between kernels (serialised); null: "
                           "nothing launched in that slot (single-launch mode: routing and "
                           "quantisation run inside the GEMM kernel)",
        "dominant_kernel": dom,
        "roofline": roofline,
        "roofline_forward": {"bound": "hbm", "alg_bytes": b_total, "achieved": fwd_gbs,
                             "peak": peak, "unit": "GB/s", "frac": fwd_gbs / peak},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "transfer": ("pinned host inputs read and pinned host output written by the "
                             "kernels in place (mapped host memory, NVLink-C2C); no staging copy")
                if in_place else "staged copies (pinned host memory not addressable in place)",
                "us_per_step": 1e3 * e2e_host_ms / e2e_steps},
        "e2e_staged": {"value": e2e_staged, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h,
                       "transfer": "one cudaMemcpyAsync of the packed pinned inputs to HBM, "
                                   "the forward on device buffers, one copy of the output back",
                       "us_per_step": 1e3 * e2e_ms / e2e_steps},
        "gpu_launches": launches * args.steps,
        "clocks": clk,
        "us_per_call_x_sm_mhz": (us_call * clk["sm_mhz"]) if clk else None,
    }
    if w.name in PUBLISHED_US:
        res["vs_baseline"] = value / (w.T / (PUBLISHED_US[w.name] * 1e-6))
    return res


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--ref-tokens", type=int, default=16)
    ap.add_argument("--ref-budget-s", type=float, default=90.0)
    ap.add_argument("--cpu-baseline-s", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--activations", default="mxfp4", choices=["mxfp4", "bf16"],
                    help="bf16: the W4A16 forward (no activation quantisation)")
    ap.add_argument("--launch", default="auto", choices=["auto", "single", "separate"],
                    help="single: route and quantise inside the GEMM kernel (2 launches per "
                         "call); separate: 4 kernels; auto: the library's choice by shape")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3

    import workloads

    w = workloads.WORKLOADS[args.workload]
    world, rank, local = dist_env()

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, w)), flush=True)
        return 0

    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    res = run_gpu(args, w, world, rank, local)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(w, args.cpu_baseline_s)
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
