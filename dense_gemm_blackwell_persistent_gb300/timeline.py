"""Timeline of one persistent-GEMM launch from a GEMM_TRACE build.

    python -c "from dense_gemm_blackwell_persistent_gb300 import _build; _build.build(variant='trace')"
    GB300_GEMM_VARIANT=trace python -m dense_gemm_blackwell_persistent_gb300.timeline --M 4096 --N 4096 --K 4096

Runs a few warm-up launches, clears the trace, runs one launch and prints,
for every trace point, the earliest / median / latest time over the CTAs
(µs from the first CTA's entry) and the per-CTA wait totals.  --json writes
the same summary to a file.

Timer reads are not ordered against barriers by the compiler: a point taken
right after a __syncthreads (teardown) can carry the time at which the
recording thread reached the barrier, not when it left it.  The epilogue's
own points (epi_end, epilogue_stores_done) bound the end of the work.
"""
from __future__ import annotations

import argparse
import json

import numpy as np
import torch

from . import (GEMM_OPT_CTA_PAIR, GEMM_OPT_DYNAMIC, GEMM_OPT_MAX_CTAS, GEMM_OPT_MULTICAST, GEMM_OPT_STREAM_K,
               GEMM_OPT_TILE_N, VARIANT,
               gemm_plan_create, gemm_plan_destroy, gemm_plan_last_grid, gemm_plan_last_launch, gemm_plan_run,
               gemm_plan_set_option, gemm_plan_trace)

POINTS = {0: "entry", 3: "first_full", 86: "epilogue_loop_done", 11: "epilogue_stores_done", 84: "producer_done",
          85: "mma_warp_done", 4: "teardown", 12: "cluster_arrived", 13: "cluster_done", 14: "tmem_dealloc", 5: "exit"}
ITEMS = {16: "mma_end", 24: "epi_start", 32: "epi_end", 40: "partial_published", 48: "reduce_done"}
TOTALS = {6: "mma_wait_full_us", 7: "producer_wait_empty_us", 8: "mma_wait_acc_empty_us",
          1: "producer_wait_response_us", 10: "mma_wait_response_us", 2: "epilogue_wait_response_us"}
PROLOGUE = {1: "barriers_initialised", 2: "tensormaps_prefetched", 3: "cluster_arrived", 4: "cluster_passed",
            5: "first_item_decoded", 6: "first_issuer_past_barrier", 7: "first_loads_issued",
            8: "mma_warp_has_tmem"}


def summarise(buf: np.ndarray, ctas: int) -> dict:
    t = buf[:ctas].astype(np.int64)
    t0 = t[:, 0][t[:, 0] > 0].min()
    out = {}

    def stats(col):
        v = t[:, col]
        v = v[v > 0]
        if v.size == 0:
            return None
        r = (v - t0) / 1e3
        return [round(float(r.min()), 2), round(float(np.median(r)), 2), round(float(r.max()), 2), int(v.size)]

    for col, name in POINTS.items():
        s = stats(col)
        if s:
            out[name] = s
    for base, name in ITEMS.items():
        for j in range(8):
            s = stats(base + j)
            if s:
                out[f"{name}[{j}]"] = s
    # SM clock: cycles and ns between first_full and each mma_end of the
    # pair leaders give the clock and the cycles per k-block of each item.
    lead = t[:, 15] > 0
    if lead.any():
        c0, n0 = t[lead, 15], t[lead, 3]
        for j in range(8):
            cj, nj = t[lead, 56 + j], t[lead, 16 + j]
            ok = (cj > 0) & (nj > 0)
            if not ok.any():
                break
            mhz = (cj[ok] - c0[ok]) / np.maximum(nj[ok] - n0[ok], 1) * 1e3
            out[f"sm_mhz_to_mma_end[{j}]"] = round(float(np.median(mhz)), 1)
            out[f"cycles_first_full_to_mma_end[{j}]"] = int(np.median(cj[ok] - c0[ok]))
    # SM cycles of the prologue steps, relative to the CTA's entry stamp
    c0 = t[:, 64]
    have = c0 > 0
    if have.any():
        for k, name in PROLOGUE.items():
            v = t[have, 64 + k]
            ok = v > 0
            if ok.any():
                d = (v[ok] - c0[have][ok]).astype(np.int64)
                out[f"cycles_to_{name}"] = [int(d.min()), int(np.median(d)), int(d.max()), int(ok.sum())]
    # SM cycles of the unit's last tile's epilogue, per epilogue warp, from
    # the warp's first step (accumulator ready): median over CTAs
    for wq in range(4):
        b = 88 + 12 * wq
        st = t[:, b]
        have = st > 0
        if not have.any():
            continue
        steps = []
        for k in range(1, 12):
            v = t[have, b + k]
            ok = v > 0
            steps.append(int(np.median(v[ok] - st[have][ok])) if ok.any() else None)
        out[f"last_epilogue_cycles_warp{wq + 2}"] = steps
    for col, name in TOTALS.items():
        v = t[:, col][t[:, col] > 0] / 1e3
        if v.size:
            out[name] = [round(float(v.min()), 2), round(float(np.median(v)), 2), round(float(v.max()), 2),
                         int(v.size)]
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--M", type=int, default=4096)
    ap.add_argument("--N", type=int, default=4096)
    ap.add_argument("--K", type=int, default=4096)
    ap.add_argument("--dtype", type=int, default=0, help="0 bf16, 1 f16")
    ap.add_argument("--out", type=int, default=0, help="0 bf16, 1 f16, 2 fp32")
    ap.add_argument("--pair", type=int, default=2)
    ap.add_argument("--tile-n", type=int, default=0)
    ap.add_argument("--stream-k", type=int, default=0)
    ap.add_argument("--dynamic", type=int, default=0, help="1: tiles handed out at run time")
    ap.add_argument("--multicast", type=int, default=-1, help="-1 auto, 0 off, 1 on")
    ap.add_argument("--max-ctas", type=int, default=0)
    ap.add_argument("--no-flush", action="store_true", help="keep the operands in L2 before the traced launch")
    ap.add_argument("--json", default="")
    a = ap.parse_args()
    if VARIANT != "trace":
        raise SystemExit("set GB300_GEMM_VARIANT=trace (and build that variant) to record a timeline")
    torch.cuda.set_device(0)
    plan = gemm_plan_create(0)
    gemm_plan_set_option(plan, GEMM_OPT_CTA_PAIR, a.pair)
    gemm_plan_set_option(plan, GEMM_OPT_TILE_N, a.tile_n)
    gemm_plan_set_option(plan, GEMM_OPT_STREAM_K, a.stream_k)
    gemm_plan_set_option(plan, GEMM_OPT_DYNAMIC, a.dynamic)
    gemm_plan_set_option(plan, GEMM_OPT_MULTICAST, a.multicast)
    gemm_plan_set_option(plan, GEMM_OPT_MAX_CTAS, a.max_ctas)
    tin = torch.bfloat16 if a.dtype == 0 else torch.float16
    tout = {0: torch.bfloat16, 1: torch.float16, 2: torch.float32}[a.out]
    A = torch.randn(a.M, a.K, device="cuda").to(tin)
    B = torch.randn(a.N, a.K, device="cuda").to(tin)
    C = torch.empty(a.M, a.N, device="cuda", dtype=tout)
    s = torch.cuda.current_stream().cuda_stream
    for _ in range(3):
        gemm_plan_run(plan, A.data_ptr(), B.data_ptr(), C.data_ptr(), a.M, a.N, a.K, a.dtype, a.out, s)
    torch.cuda.synchronize()
    gemm_plan_trace(plan)
    if not a.no_flush:
        torch.empty(512 << 20, dtype=torch.uint8, device="cuda").zero_()   # evict A, B, C from L2
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    gemm_plan_run(plan, A.data_ptr(), B.data_ptr(), C.data_ptr(), a.M, a.N, a.K, a.dtype, a.out, s)
    e1.record()
    torch.cuda.synchronize()
    buf = gemm_plan_trace(plan)
    res = summarise(buf, gemm_plan_last_grid(plan))
    # The launch as CUDA events see it, beside the span the CTAs themselves
    # stamped (first entry to last exit): the difference is launch and
    # completion latency outside the kernel's code.
    res["event_us"] = round(e0.elapsed_time(e1) * 1e3, 2)
    launch = gemm_plan_last_launch(plan)
    print(f"{a.M}x{a.N}x{a.K} unit={launch['ctas_per_unit']} tile_n={launch['tile_n']} ctas={launch['ctas']} "
          f"stream_k={a.stream_k} l2={'warm' if a.no_flush else 'flushed'}: "
          "[earliest, median, latest] µs over CTAs, count")
    for k, v in res.items():
        print(f"  {k:26s} {v}")
    if a.json:
        with open(a.json, "w") as f:
            json.dump(res, f, indent=1)
    gemm_plan_destroy(plan)


if __name__ == "__main__":
    main()
