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

    plan = g.gemm_plan_create(local)
    if args.cta_pair:
        g.gemm_plan_set_option(plan, g.GEMM_OPT_CTA_PAIR, args.cta_pair)
    g.gemm_plan_set_option(plan, g.GEMM_OPT_DYNAMIC, args.dynamic)
    if args.group_m:
        g.gemm_plan_set_option(plan, g.GEMM_OPT_GROUP_M, args.group_m)
    if args.tile_n:
        g.gemm_plan_set_option(plan, g.GEMM_OPT_TILE_N, args.tile_n)
    g.gemm_plan_set_option(plan, g.GEMM_OPT_MULTICAST, args.multicast)
    g.gemm_plan_set_option(plan, g.GEMM_OPT_STREAM_K, args.stream_k)

    A_cpu, B_cpu = wl.make_inputs(w)
    A, B = A_cpu.cuda(), B_cpu.cuda()
    out_t = wl.TORCH_DTYPES[w.out_dtype]
    C = torch.empty((w.M, w.N), dtype=out_t, device="cuda")
    flush = None if args.no_flush else torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream

    def step():
        g.gemm_plan_run(plan, A.data_ptr(), B.data_ptr(), C.data_ptr(), w.M, w.N, w.K, w.dtype, w.out_dtype, sp)

    for _ in range(max(3, args.warmup)):
        if flush is not None:
            flush.zero_()
        step()
    torch.cuda.synchronize()
    if g.gemm_plan_status(plan) != 0:
        raise SystemExit("device status error during warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.25)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    status = g.gemm_plan_status(plan)
    if status != 0:
        raise SystemExit(f"device status {status} after the timed region")
    launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    value, ms_per_step = aggregate(world, w.flops, args.steps, sum(launch_ms))
    avg_launch_ms = statistics.mean(launch_ms)
    achieved = w.flops / (avg_launch_ms / 1e3) / 1e12

    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    peak_note = f"{peak_src}: MEASURED_PEAKS bf16_tflops (burst, cuBLAS 8192^3)"
    if w.dtype in wl.FP8:
        # no measured fp8 figure: the bf16 one times the nominal dense ratio 4.5 / 2.25
        peak *= 2.0
        peak_note += " x 2 (nominal fp8:bf16 dense ratio)"
    timed_launch = g.gemm_plan_last_launch(plan)   # before the e2e runs launch other shapes
    traffic = recorded_traffic(w.name, timed_launch)

    extra = {}
    ref_call, ref_how = None, None
    if w.dtype in wl.FP8:
        one = torch.ones((), dtype=torch.float32, device="cuda")
        if hasattr(torch, "_scaled_mm"):
            ref_call = lambda: torch._scaled_mm(A, B.t(), scale_a=one, scale_b=one, out_dtype=out_t)
            ref_how = "torch._scaled_mm(A, B.t(), unit scales, out bf16)"
    elif w.out_dtype == w.dtype:
        Bt = B.t()
        ref_call = lambda: torch.matmul(A, Bt)
        ref_how = "torch.matmul(A, B.t())"
    if not args.no_cublas and rank == 0 and ref_call is not None:
        try:
            for _ in range(5):
                ref_call()
            # Same protocol as the timed steps: events around each launch on
            # the stream, no host synchronisation inside the loop (a host
            # wait per run would put the next launch's host-side latency
            # inside its events whenever no flush is queued ahead of it).
            cs = [torch.cuda.Event(enable_timing=True) for _ in range(50)]
            ce = [torch.cuda.Event(enable_timing=True) for _ in range(50)]
            for i in range(50):
                if flush is not None:
                    flush.zero_()
                cs[i].record(stream)
                ref_call()
                ce[i].record(stream)
            torch.cuda.synchronize()
            cm = statistics.mean(a.elapsed_time(b) for a, b in zip(cs, ce))
            l2 = "L2 flushed" if flush is not None else "L2 not flushed"
            extra["cublas_reference"] = {"value": w.flops / (cm / 1e3) / 1e12, "unit": "TFLOP/s", "ms": cm,
                                         "how": f"{ref_how}, same inputs, same process, 50 runs, {l2}"}
        except RuntimeError as e:   # a torch build without this fp8 path: no reference line
            extra["cublas_reference"] = {"unavailable": str(e).splitlines()[0][:200]}

    # Context for the roofline: the tensor cores' own rate, measured by a
    # stream of back-to-back MMAs of this kernel's shape with no loads, on
    # every SM, right after the timed region (outside it).
    mma_probe = None
    if rank == 0 and not args.no_probe:
        r = g.gemm_probe_mma_rate(w.dtype, args.cta_pair or 2, 1 << 16)
        sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
        mma_probe = {"tflops": r["tflops"], "sm_mhz": r["sm_mhz"], "flop_per_clk_per_sm": r["flop_per_clk_per_sm"],
                     "frac": achieved / r["tflops"],
                     "peak_at_max_clock_tflops":
                         r["flop_per_clk_per_sm"] * sms * float(peaks.get("sm_max_mhz", 2070.0)) / 1e6,
                     "how": "gemm_probe_mma_rate: 65536 back-to-back tcgen05.mma per SM, operands in shared memory, "
                            "no loads; frac = achieved / tflops"}

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
               "how": "gemm_plan_run_host: pinned host A,B in, host C out, row chunks with copies in, products and copies back overlapped on the plan's streams, sync per step, "
                      f"host wall clock, {args.e2e_steps} steps"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, wl.as_bits(A_cpu), wl.as_bits(B_cpu), args.cpu_seconds)

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
                       "tile_per_mma": f"{128 * (args.cta_pair or 2)}x{timed_launch['tile_n']}x"
                                       f"{128 // wl.ELEM_BYTES[w.dtype]}",
                       "vs_baseline_ref": "pages' 293.6 TFLOP/s, Mojo part-2 kernel 4 on B200 (context)"},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_source": peak_note, "mma_probe": mma_probe},
            "clocks": clocks,
            "gpu_launches": args.steps,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "timed_wall_s": wall,
            "launch_ms": {"mean": avg_launch_ms, "min": min(launch_ms), "median": statistics.median(launch_ms)},
        }
        line.update(extra)
        print(json.dumps(line), flush=True)
    g.gemm_plan_destroy(plan)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
