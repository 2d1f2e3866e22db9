#!/usr/bin/env python3
"""Throughput of the GB300 dense GEMM C = A·Bᵀ (TFLOP/s) and its roofline fraction.

One step = one C = A·Bᵀ over the whole workload (one launch of the persistent
kernel).  Default workload: bf16 M=N=K=4096, bf16 out, A and B ~ N(0,1),
seed 1 (the shape the Mojo Blackwell series is measured on).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Timing: K steps, each bracketed by CUDA events on the launching stream, with
L2 flushed (a 512 MiB device write) before every step, outside the events.
Under torchrun (N > 1) every rank runs an independent replica of the same
workload on its own GPU (the product shards into independent problems; there
is no data-path collective); value = all ranks' FLOPs ÷ the slowest rank's
time.  Rank 0 prints one JSON line.

--impl reference times the CPU oracle (fp64 triple loop, test
infrastructure) on the host cores, each step a bounded row-block sample of
the same workload.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

PAGES_B200_TFLOPS = 293.6   # bf16 4096^3, Mojo part-2 kernel 4 on B200 (context, another machine)
METRIC = "GEMM TFLOP/s on 1 GB300 (bf16 4096³) and % of dense tensor-core roofline"
KERNEL_NAME = "gemm_tn_persistent"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="gemm_4096_bf16", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cublas", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-flush", action="store_true", help="do not flush L2 between steps")
    ap.add_argument("--cta-pair", type=int, default=0, help="force 1 or 2 (0 = library default)")
    ap.add_argument("--group-m", type=int, default=0)
    ap.add_argument("--tile-n", type=int, default=0, help="force the tile width (0 = library choice)")
    ap.add_argument("--multicast", type=int, default=-1, help="-1 auto, 0 off, 1 on (CTA pairs only)")
    ap.add_argument("--stream-k", type=int, default=0, help="1: stream-K tail")
    ap.add_argument("--dynamic", type=int, default=-1, help="-1 auto, 0 static, 1 hand out the partial wave, 2 every tile")
    ap.add_argument("--no-probe", action="store_true", help="skip the tensor-core issue-rate probe")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU-baseline sample budget")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the context lines (back-to-back run, other workloads, sustained runs)")
    ap.add_argument("--sustained-s", type=float, default=4.0, help="seconds of each sustained run (0 = none)")
    return ap.parse_args()


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, local, world


def max_over_ranks(x: float) -> float:
    """Largest value of `x` over all ranks (the slowest rank's time); x itself
    when not running under torch.distributed."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(world: int, flops_per_step: float, steps: int, local_ms_total: float):
    """Whole-job throughput: every rank runs `steps` steps of its own replica;
    value = all ranks' FLOPs ÷ the slowest rank's time (TFLOP/s), and the
    per-step time of that slowest rank (ms)."""
    slowest = max_over_ranks(local_ms_total)
    return world * flops_per_step * steps / (slowest / 1e3) / 1e12, slowest / steps


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# Device-side sources: what a launch of the kernel executes.  The host side
# (gemm_api.cu) only chooses the launch shape, which traffic records carry
# separately.
DEVICE_SOURCES = ("gemm_kernel.cuh", "kernel_table.h", "kernels_inst.cu", "ptx.cuh", "schedule.h")


def _code_only(text: str) -> str:
    """Source text without comments, trailing spaces and blank lines: a
    comment edit does not change the kernel the counters were taken on."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", line).rstrip() for line in text.splitlines())
    return "\n".join(line for line in lines if line)


def source_digest() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_gemm_blackwell_persistent_gb300", "csrc")
    for name in DEVICE_SOURCES:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def launch_key(launch: dict) -> str:
    return " ".join(f"{k}={launch[k]}" for k in ("ctas", "ctas_per_unit", "tile_n", "dp_waves", "sk_tiles"))


def recorded_traffic(workload: str, launch: dict = None):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current device code (its digest line must match) and, when `launch`
    is given, with the same launch shape; else None."""
    path = os.path.join(ROOT, "profiles", f"traffic_{KERNEL_NAME}_{workload}.txt")
    try:
        fields = dict(line.split(":", 1) for line in open(path) if ":" in line and not line.startswith("#"))
    except OSError:
        return None
    if fields.get("source_digest", "").strip() != source_digest():
        return None
    if launch is not None and fields.get("launch", "").strip() != launch_key(launch):
        return None
    try:
        return int(fields["dram_bytes_per_launch"].strip())
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        return summarise_clocks(self.lines)


def summarise_clocks(lines):
    """Median SM clock, maximum clock, throttle reasons seen and peak power from
    `nvidia-smi --query-gpu=<ClockSampler.QUERY> --format=csv,noheader,nounits`
    lines; lines that do not parse (a header, [N/A] fields) are skipped."""
    sm, smax, power, reasons = [], None, [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            clock, top, watts = float(parts[1]), float(parts[2]), float(parts[3])
        except ValueError:
            continue
        sm.append(clock)
        smax = top
        power.append(watts)
        for nm, v in zip(names, parts[5:9]):
            if v.lower() == "active":
                reasons.add(nm)
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
            "reasons": sorted(reasons), "samples": len(sm),
            "power_w_max": max(power) if power else None}


def cpu_baseline(w: wl.Workload, A_bits, B_bits, budget_s: float):
    """The oracle as it stands on a row-block sample of the workload.

    Two short calibration calls separate the oracle's fixed cost (decoding
    all of B) from its per-row cost, so the timed sample lasts about
    `budget_s` seconds."""
    import oracle
    o = oracle.default()
    times = []
    for r in (1, min(w.M, 9)):
        t0 = time.perf_counter()
        o.gemm(A_bits[:r], B_bits, w.dtype)
        times.append((r, time.perf_counter() - t0))
    (r1, t1), (r2, t2) = times
    per_row = max((t2 - t1) / max(r2 - r1, 1), 1e-6)
    fixed = max(t1 - per_row * r1, 0.0)
    rows = int(max(1, min(w.M, (budget_s - fixed) / per_row)))
    t0 = time.perf_counter()
    o.gemm(A_bits[:rows], B_bits, w.dtype)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * w.N * w.K
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": o.max_threads(), "kind": "oracle",
            "sample": f"rows 0..{rows - 1} of A against all of B ({rows}x{w.N}x{w.K}), {dt:.1f} s, "
                      f"fp64 triple loop incl. operand decode"}


def cpu_single_thread_256():
    """The oracle on one thread for the 256³ workload (whole product)."""
    import oracle
    w1 = wl.WORKLOADS["gemm_256_f32out"]
    A, B = wl.make_inputs(w1)
    Ab, Bb = wl.as_bits(A), wl.as_bits(B)
    oracle.gemm(Ab[:8], Bb, w1.dtype, threads=1)
    t0 = time.perf_counter()
    oracle.gemm(Ab, Bb, w1.dtype, threads=1)
    dt = time.perf_counter() - t0
    return {"value": w1.flops / dt / 1e12, "unit": "TFLOP/s", "seconds": dt, "cores": 1,
            "sample": "the whole 256x256x256 product, fp64 triple loop incl. operand decode, 1 thread"}


def run_reference(args, w: wl.Workload):
    rank, _, world = dist_info()
    if world > 1 and rank != 0:
        return
    import oracle
    o = oracle.default()
    A, B = wl.make_inputs(w)
    A_bits, B_bits = wl.as_bits(A), wl.as_bits(B)
    total_budget = 150.0
    per_step = min(30.0, total_budget / max(1, args.steps + args.warmup))
    t0 = time.perf_counter()
    o.gemm(A_bits[:1], B_bits, w.dtype)
    one = time.perf_counter() - t0
    rows = int(max(1, min(w.M, per_step / max(one, 1e-6))))
    for _ in range(args.warmup):
        o.gemm(A_bits[:rows], B_bits, w.dtype)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        o.gemm(A_bits[:rows], B_bits, w.dtype)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.mean(times)
    value = 2.0 * rows * w.N * w.K / (ms / 1e3) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "in": wl.DTYPE_NAMES[w.dtype],
                   "out": wl.DTYPE_NAMES[w.out_dtype], "sample_rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": o.max_threads(), "kind": "oracle",
                         "sample": f"each step: rows 0..{rows - 1} of A against all of B "
                                   f"({rows}x{w.N}x{w.K}), fp64 triple loop incl. operand decode"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# The other workloads of the benchmark set, each timed briefly in the same
# process after the main one (their lines go under "other_workloads").
OTHER_WORKLOADS = ["gemm_256_f32out", "gemm_1024x4096x4096_f16", "gemm_ragged_4000x3000x5000", "gemm_8192_bf16",
                   "gemm_4096_e4m3"]
SUSTAINED_WORKLOADS = ["gemm_4096_bf16", "gemm_8192_bf16"]


def make_plan(g, args, device):
    plan = g.gemm_plan_create(device)
    if args.cta_pair:
        g.gemm_plan_set_option(plan, g.GEMM_OPT_CTA_PAIR, args.cta_pair)
    g.gemm_plan_set_option(plan, g.GEMM_OPT_DYNAMIC, args.dynamic)
    if args.group_m:
        g.gemm_plan_set_option(plan, g.GEMM_OPT_GROUP_M, args.group_m)
    if args.tile_n:
        g.gemm_plan_set_option(plan, g.GEMM_OPT_TILE_N, args.tile_n)
    g.gemm_plan_set_option(plan, g.GEMM_OPT_MULTICAST, args.multicast)
    g.gemm_plan_set_option(plan, g.GEMM_OPT_STREAM_K, args.stream_k)
    return plan


def kernel_clock(records):
    """SM clock of the timed launches from the plan's clock log: per launch
    cycles ÷ ns of its first CTA's lifetime, summarised."""
    mhz = [c / ns * 1e3 for c, ns in records if ns > 0]
    if not mhz:
        return None
    return {"sm_mhz_median": statistics.median(mhz), "sm_mhz_min": min(mhz), "sm_mhz_max": max(mhz),
            "launches": len(mhz),
            "how": "clock64 and %globaltimer at entry and exit of each launch's first CTA (GEMM_OPT_CLOCK_LOG)"}


def tensor_peak(peaks, dtype):
    """The measured dense peak for the operand type, and where it comes from."""
    peak = float(peaks["bf16_tflops"])
    note = "MEASURED_PEAKS bf16_tflops (burst, cuBLAS 8192^3)"
    if dtype in wl.FP8:
        # no measured fp8 figure: the bf16 one times the nominal dense ratio 4.5 / 2.25
        peak *= 2.0
        note += " x 2 (nominal fp8:bf16 dense ratio)"
    return peak, note


def roofline(w, achieved_tflops, mean_ms, peaks, peak_src, probe, sms, clock):
    """Roofline of one launch: the bound is the slower of the FLOPs at the
    measured tensor peak and the compulsory bytes at the measured HBM copy
    bandwidth; achieved and peak are in that bound's unit.  Also the fraction
    of the tensor cores' own rate at the maximum SM clock and at the clock the
    launches ran at (issue-rate probe × SMs × clock)."""
    peak, note = tensor_peak(peaks, w.dtype)
    hbm = float(peaks["hbm_gbs"])
    t_flop = w.flops / (peak * 1e12)
    t_mem = w.compulsory_bytes / (hbm * 1e9)
    bound = "tensor" if t_flop >= t_mem else "hbm"
    if bound == "tensor":
        out = {"bound": bound, "achieved": achieved_tflops, "peak": peak, "unit": "TFLOP/s",
               "frac": achieved_tflops / peak}
    else:
        gbs = w.compulsory_bytes / (mean_ms / 1e3) / 1e9
        out = {"bound": bound, "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm}
    out["peak_source"] = f"{peak_src}: " + (note if bound == "tensor" else "MEASURED_PEAKS hbm_gbs (copy)")
    out["terms_us"] = {"flops_at_peak": t_flop * 1e6, "compulsory_bytes_at_hbm": t_mem * 1e6}
    if probe is not None:
        per_clk = probe["flop_per_clk_per_sm"]
        at_max = per_clk * sms * float(peaks.get("sm_max_mhz", 2070.0)) / 1e6
        out["peak_clock_tflops"] = at_max
        out["frac_peak_clock"] = achieved_tflops / at_max
        if clock is not None:
            at_run = per_clk * sms * clock["sm_mhz_median"] / 1e6
            out["kernel_clock_tflops"] = at_run
            out["frac_kernel_clock"] = achieved_tflops / at_run
        out["peak_clock_how"] = ("tcgen05.mma issue-rate probe (FLOP per SM clock, measured) x SMs x "
                                 "MEASURED_PEAKS sm_max_mhz; kernel clock: the timed launches' own")
    return out


def cublas_call(torch, w, A, B, out_t):
    """The cuBLAS reference for workload w (same inputs, same output type), or
    (None, reason)."""
    if w.dtype in wl.FP8:
        if not hasattr(torch, "_scaled_mm"):
            return None, "torch._scaled_mm missing"
        one = torch.ones((), dtype=torch.float32, device="cuda")
        return (lambda: torch._scaled_mm(A, B.t(), scale_a=one, scale_b=one, out_dtype=out_t)), \
            "torch._scaled_mm(A, B.t(), unit scales)"
    Bt = B.t()
    if w.out_dtype == w.dtype:
        return (lambda: torch.matmul(A, Bt)), "torch.matmul(A, B.t())"
    return (lambda: torch.mm(A, Bt, out_dtype=out_t)), "torch.mm(A, B.t(), out_dtype=float32)"


def time_cublas(torch, w, call, how, stream, flush, runs=50):
    try:
        for _ in range(5):
            call()
        cs = [torch.cuda.Event(enable_timing=True) for _ in range(runs)]
        ce = [torch.cuda.Event(enable_timing=True) for _ in range(runs)]
        # Same protocol as the timed steps: events around each launch on the
        # stream, no host synchronisation inside the loop.
        for i in range(runs):
            if flush is not None:
                flush.zero_()
            cs[i].record(stream)
            call()
            ce[i].record(stream)
        torch.cuda.synchronize()
    except (RuntimeError, NotImplementedError, TypeError) as e:   # no such path in this torch build
        return {"unavailable": f"{how}: " + str(e).splitlines()[0][:200]}
    cm = statistics.mean(a.elapsed_time(b) for a, b in zip(cs, ce))
    l2 = "L2 flushed" if flush is not None else "L2 not flushed"
    return {"value": w.flops / (cm / 1e3) / 1e12, "unit": "TFLOP/s", "ms": cm,
            "how": f"{how}, same inputs, same process, {runs} runs, {l2}"}


def time_launches(torch, g, plan, w, A, B, C, stream, steps, warmup, flush, barrier=None):
    """CUDA events around each of `steps` launches on `stream` (after `warmup`
    untimed ones), L2 flushed before each step when `flush` is a buffer; the
    timed loop is bracketed by `barrier()` (all ranks) and a device
    synchronisation on both sides.  Returns the per-launch times (ms), the
    clock log of the timed launches and the host wall time of the timed loop."""
    sp = stream.cuda_stream

    def step():
        g.gemm_plan_run(plan, A.data_ptr(), B.data_ptr(), C.data_ptr(), w.M, w.N, w.K, w.dtype, w.out_dtype, sp)

    for _ in range(max(3, warmup)):
        if flush is not None:
            flush.zero_()
        step()
    torch.cuda.synchronize()
    if g.gemm_plan_status(plan) != 0:
        raise SystemExit(f"{w.name}: device status error during warm-up")
    g.gemm_plan_set_option(plan, g.GEMM_OPT_CLOCK_LOG, steps)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    if barrier is not None:
        barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if barrier is not None:
        barrier()
    status = g.gemm_plan_status(plan)
    if status != 0:
        raise SystemExit(f"{w.name}: device status {status} after the timed region")
    records = g.gemm_plan_clock_log(plan, capacity=steps)
    g.gemm_plan_set_option(plan, g.GEMM_OPT_CLOCK_LOG, 0)
    return [s.elapsed_time(e) for s, e in zip(starts, ends)], records, wall


def other_workload_line(torch, g, args, name, peaks, peak_src, probe_rates, sms, stream, flush, local):
    """Short flushed run of one more workload: TFLOP/s, roofline, kernel clock,
    launch shape and the cuBLAS line on the same inputs."""
    w = wl.WORKLOADS[name]
    A_cpu, B_cpu = wl.make_inputs(w)
    A, B = A_cpu.cuda(), B_cpu.cuda()
    out_t = wl.TORCH_DTYPES[w.out_dtype]
    C = torch.empty((w.M, w.N), dtype=out_t, device="cuda")
    plan = make_plan(g, args, local)
    try:
        steps = 200 if w.flops < 1e11 else 50
        ms, records, _ = time_launches(torch, g, plan, w, A, B, C, stream, steps, 5, flush)
        launch = g.gemm_plan_last_launch(plan)
    finally:
        g.gemm_plan_destroy(plan)
    mean_ms = statistics.mean(ms)
    achieved = w.flops / (mean_ms / 1e3) / 1e12
    clock = kernel_clock(records)
    line = {"value": achieved, "unit": "TFLOP/s", "steps": steps, "ms_mean": mean_ms, "ms_min": min(ms),
            "ms_median": statistics.median(ms), "launch": launch, "kernel_clock": clock,
            "roofline": roofline(w, achieved, mean_ms, peaks, peak_src, probe_rates.get(w.dtype), sms, clock),
            "config": {"M": w.M, "N": w.N, "K": w.K, "in": wl.DTYPE_NAMES[w.dtype],
                       "out": wl.DTYPE_NAMES[w.out_dtype], "inputs": w.describe()}}
    line["roofline"]["traffic"] = recorded_traffic(w.name, launch)
    if not args.no_cublas:
        call, how = cublas_call(torch, w, A, B, out_t)
        line["cublas_reference"] = time_cublas(torch, w, call, how, stream, flush) if call else {"unavailable": how}
    return line


def sustained_line(torch, g, args, name, seconds, stream, local):
    """Back-to-back launches for about `seconds` (no flush: MEASURED_PEAKS'
    sustained method, operands resident), one pair of events around the
    whole loop; the launches' own clock and nvidia-smi's beside it."""
    w = wl.WORKLOADS[name]
    A_cpu, B_cpu = wl.make_inputs(w)
    A, B = A_cpu.cuda(), B_cpu.cuda()
    C = torch.empty((w.M, w.N), dtype=wl.TORCH_DTYPES[w.out_dtype], device="cuda")
    plan = make_plan(g, args, local)
    sp = stream.cuda_stream
    try:
        def step():
            g.gemm_plan_run(plan, A.data_ptr(), B.data_ptr(), C.data_ptr(), w.M, w.N, w.K, w.dtype, w.out_dtype,
                            sp)
        for _ in range(10):
            step()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(20):
            step()
        torch.cuda.synchronize()
        per = (time.perf_counter() - t0) / 20
        n = max(20, int(seconds / per))
        g.gemm_plan_set_option(plan, g.GEMM_OPT_CLOCK_LOG, n)
        sampler = ClockSampler(local)
        sampler.start()
        time.sleep(0.25)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(n):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        smi = sampler.stop()
        if g.gemm_plan_status(plan) != 0:
            raise SystemExit(f"{name}: device status error in the sustained run")
        records = g.gemm_plan_clock_log(plan, capacity=n)
    finally:
        g.gemm_plan_destroy(plan)
    ms = ev0.elapsed_time(ev1)
    line = {"value": w.flops * n / (ms / 1e3) / 1e12, "unit": "TFLOP/s", "launches": n, "seconds": ms / 1e3,
            "kernel_clock": kernel_clock(records), "clocks": smi,
            "how": "back-to-back launches, operands resident (no flush), events around the whole loop"}
    if not args.no_cublas:
        # cuBLAS the same way, right after: same inputs, as many launches
        call, how = cublas_call(torch, w, A, B, wl.TORCH_DTYPES[w.out_dtype])
        try:
            for _ in range(10):
                call()
            torch.cuda.synchronize()
            sampler = ClockSampler(local)
            sampler.start()
            time.sleep(0.25)
            ev0.record(stream)
            for _ in range(n):
                call()
            ev1.record(stream)
            torch.cuda.synchronize()
            smi_ref = sampler.stop()
            ms_ref = ev0.elapsed_time(ev1)
            line["cublas_reference"] = {"value": w.flops * n / (ms_ref / 1e3) / 1e12, "unit": "TFLOP/s",
                                        "launches": n, "seconds": ms_ref / 1e3, "clocks": smi_ref,
                                        "how": f"{how}, back to back right after, same inputs"}
        except (RuntimeError, NotImplementedError, TypeError) as e:
            line["cublas_reference"] = {"unavailable": f"{how}: " + str(e).splitlines()[0][:200]}
    return line


def back_to_back_line(torch, g, args, w, A, B, C, out_t, stream, local, n=200):
    """The same workload with L2 left warm: n launches enqueued back to back
    between two events (no host gap inside; the library's launches overlap
    their set-up with the previous launch's end), time ÷ n; cuBLAS the same
    way on the same inputs."""
    plan = make_plan(g, args, local)
    sp = stream.cuda_stream
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    try:
        for _ in range(10):
            g.gemm_plan_run(plan, A.data_ptr(), B.data_ptr(), C.data_ptr(), w.M, w.N, w.K, w.dtype, w.out_dtype, sp)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n):
            g.gemm_plan_run(plan, A.data_ptr(), B.data_ptr(), C.data_ptr(), w.M, w.N, w.K, w.dtype, w.out_dtype, sp)
        e1.record(stream)
        torch.cuda.synchronize()
        if g.gemm_plan_status(plan) != 0:
            raise SystemExit(f"{w.name}: device status error in the back-to-back run")
    finally:
        g.gemm_plan_destroy(plan)
    ms = e0.elapsed_time(e1) / n
    line = {"value": w.flops / (ms / 1e3) / 1e12, "unit": "TFLOP/s", "ms_per_launch": ms, "launches": n,
            "how": "launches back to back between two events, operands resident in L2 (no flush), "
                   "programmatic dependent launch on"}
    if not args.no_cublas:
        call, how = cublas_call(torch, w, A, B, out_t)
        try:
            for _ in range(10):
                call()
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(n):
                call()
            e1.record(stream)
            torch.cuda.synchronize()
            ms_ref = e0.elapsed_time(e1) / n
            line["cublas_reference"] = {"value": w.flops / (ms_ref / 1e3) / 1e12, "unit": "TFLOP/s",
                                        "ms_per_launch": ms_ref, "how": f"{how}, the same way"}
        except (RuntimeError, NotImplementedError, TypeError) as e:
            line["cublas_reference"] = {"unavailable": f"{how}: " + str(e).splitlines()[0][:200]}
    return line


def main():
    args = parse_args()
    w = wl.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
        return
    rank, local, world = dist_info()

    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    import dense_gemm_blackwell_persistent_gb300 as g

    plan = make_plan(g, args, local)
    A_cpu, B_cpu = wl.make_inputs(w)
    A, B = A_cpu.cuda(), B_cpu.cuda()
    out_t = wl.TORCH_DTYPES[w.out_dtype]
    C = torch.empty((w.M, w.N), dtype=out_t, device="cuda")
    flush = None if args.no_flush else torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count

    barrier = torch.distributed.barrier if world > 1 else None
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.25)
    launch_ms, records, wall = time_launches(torch, g, plan, w, A, B, C, stream, args.steps, args.warmup, flush,
                                             barrier)
    clocks = sampler.stop()
    clocks["in_kernel"] = kernel_clock(records)
    value, ms_per_step = aggregate(world, w.flops, args.steps, sum(launch_ms))
    avg_launch_ms = statistics.mean(launch_ms)
    achieved = w.flops / (avg_launch_ms / 1e3) / 1e12
    timed_launch = g.gemm_plan_last_launch(plan)   # before the e2e runs launch other shapes

    peaks, peak_src = load_peaks()
    # The tensor cores' own rate, measured by a stream of back-to-back MMAs of
    # this kernel's shape with no loads, on every SM, after the timed region
    # (outside it): per operand width, for the roofline at a given clock.
    probe_rates = {}
    if rank == 0 and not args.no_probe:
        for dt in sorted({w.dtype, wl.BF16, wl.F16, wl.E4M3}):
            probe_rates[dt] = g.gemm_probe_mma_rate(dt, args.cta_pair or 2, 1 << 16)
    probe = probe_rates.get(w.dtype)
    roof = roofline(w, achieved, avg_launch_ms, peaks, peak_src, probe, sms, clocks["in_kernel"])
    roof["traffic"] = recorded_traffic(w.name, timed_launch)
    if probe is not None:
        roof["mma_probe"] = {"tflops": probe["tflops"], "sm_mhz": probe["sm_mhz"],
                             "flop_per_clk_per_sm": probe["flop_per_clk_per_sm"], "frac": achieved / probe["tflops"],
                             "how": "gemm_probe_mma_rate: 65536 back-to-back tcgen05.mma per SM, operands in "
                                    "shared memory, no loads; frac = achieved / tflops at the probe's own clock"}

    extra = {}
    if not args.no_cublas and rank == 0:
        call, how = cublas_call(torch, w, A, B, out_t)
        extra["cublas_reference"] = time_cublas(torch, w, call, how, stream, flush) if call else {"unavailable": how}

    e2e = None
    if not args.no_e2e:
        Ah, Bh = A_cpu.pin_memory(), B_cpu.pin_memory()
        Ch = torch.empty((w.M, w.N), dtype=out_t).pin_memory()
        g.gemm_plan_run_host(plan, Ah.data_ptr(), Bh.data_ptr(), Ch.data_ptr(), w.M, w.N, w.K, w.dtype,
                             w.out_dtype, sp)
        es = []
        for _ in range(args.e2e_steps):
            t0 = time.perf_counter()
            g.gemm_plan_run_host(plan, Ah.data_ptr(), Bh.data_ptr(), Ch.data_ptr(), w.M, w.N, w.K, w.dtype,
                                 w.out_dtype, sp)
            es.append(time.perf_counter() - t0)
        e2e_value, _ = aggregate(world, w.flops, args.e2e_steps, 1e3 * sum(es))
        e2e = {"value": e2e_value, "unit": "TFLOP/s",
               "h2d_bytes_per_step": (w.M + w.N) * w.K * wl.ELEM_BYTES[w.dtype],
               "d2h_bytes_per_step": w.M * w.N * wl.ELEM_BYTES[w.out_dtype],
               "how": "gemm_plan_run_host: pinned host A,B in, host C out, row chunks with copies in, products and "
                      "copies back overlapped on the plan's streams, sync per step, "
                      f"host wall clock, {args.e2e_steps} steps"}
    g.gemm_plan_destroy(plan)

    # Context lines, outside the timed region (rank 0 only): the same
    # workload back to back with L2 left warm, the other workloads of the
    # benchmark set, and seconds-long back-to-back runs at the power limit.
    if rank == 0 and not args.no_extra:
        extra["back_to_back"] = back_to_back_line(torch, g, args, w, A, B, C, out_t, stream, local)
        del A, B, C
        others = {}
        for name in OTHER_WORKLOADS:
            if name != w.name:
                others[name] = other_workload_line(torch, g, args, name, peaks, peak_src, probe_rates, sms, stream,
                                                   flush, local)
        extra["other_workloads"] = others
        if args.sustained_s > 0:
            extra["sustained"] = {name: sustained_line(torch, g, args, name, args.sustained_s, stream, local)
                                  for name in SUSTAINED_WORKLOADS}
            extra["sustained"]["reference"] = {"bf16_tflops_sustained": peaks.get("bf16_tflops_sustained"),
                                               "source": f"{peak_src}: MEASURED_PEAKS (cuBLAS 8192^3, 4 s)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, wl.as_bits(A_cpu), wl.as_bits(B_cpu), args.cpu_seconds)
        cpu["single_thread_256"] = cpu_single_thread_256()

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": value / PAGES_B200_TFLOPS if w.name == "gemm_4096_bf16" else None,
            "dtype": wl.DTYPE_NAMES[w.dtype], "data": "synthetic",
            "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "in": wl.DTYPE_NAMES[w.dtype],
                       "out": wl.DTYPE_NAMES[w.out_dtype], "accumulate": "f32",
                       "inputs": w.describe(), "parallelism": f"replicas x{world}",
                       "l2": "not flushed" if args.no_flush else "flushed before every step (512 MiB write)",
                       "launch": timed_launch,
                       "tile_per_mma": f"{128 * min(timed_launch['ctas_per_unit'], 2)}x{timed_launch['tile_n']}x"
                                       f"{128 // wl.ELEM_BYTES[w.dtype]}",
                       "vs_baseline_ref": "pages' 293.6 TFLOP/s, Mojo part-2 kernel 4 on B200 (context)"},
            "roofline": roof,
            "clocks": clocks,
            "gpu_launches": args.steps,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "timed_wall_s": wall,
            "launch_ms": {"mean": avg_launch_ms, "min": min(launch_ms), "median": statistics.median(launch_ms)},
        }
        line.update(extra)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
