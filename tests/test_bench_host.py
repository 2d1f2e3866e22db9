"""bench.py host logic without a GPU: the multi-rank aggregation over a real
two-rank gloo process group, and the reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r ran its 10 steps in (r + 1) * 100 ms; the job is timed by the slowest rank
        value, ms_per_step = bench.aggregate(world, 1e12, 10, (rank + 1) * 100.0)
        q.put((rank, bench.dist_info(), value, ms_per_step, bench.max_over_ranks(float(rank))))
    finally:
        dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, info, value, ms_per_step, mx in got:
        assert info == (rank, rank, 2)
        # 2 ranks × 10 steps × 1e12 FLOP over the slowest rank's 0.2 s
        assert value == pytest.approx(2 * 10 * 1e12 / 0.2 / 1e12)
        assert ms_per_step == pytest.approx(20.0)
        assert mx == 1.0


def test_aggregate_single_process():
    sys.path.insert(0, ROOT)
    import bench
    value, ms = bench.aggregate(1, 2e12, 4, 400.0)
    assert value == pytest.approx(4 * 2e12 / 0.4 / 1e12) and ms == pytest.approx(100.0)


def test_reference_arm_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "gemm_256_f32out", "--steps", "2", "--warmup", "0"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"] == "gemm_256_f32out"


def test_clock_summary_from_nvidia_smi_lines():
    sys.path.insert(0, ROOT)
    import bench
    lines = [
        "index, clocks.current.sm [MHz], clocks.max.sm [MHz], power.draw [W], ...",   # a header: skipped
        "0, 2070, 2070, 640.12, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1725, 2070, 1372.50, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 1800, 2070, 1100.00, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, [N/A], 2070, [N/A], [N/A], [N/A], [N/A], [N/A], [N/A]",                      # unreadable: skipped
        "0, 2070",                                                                          # truncated: skipped
    ]
    c = bench.summarise_clocks(lines)
    assert c == {"sm_mhz": 1800.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3,
                 "power_w_max": 1372.5}
    throttled = bench.summarise_clocks([
        "0, 1500, 2070, 900, 0x8, Active, Not Active, Active, Not Active"])
    assert throttled["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert bench.summarise_clocks([])["sm_mhz"] is None


def test_roofline_bound_is_the_slower_term():
    """The bound is whichever is slower: the FLOPs at the measured tensor peak
    or the compulsory bytes at the measured copy bandwidth; achieved and peak
    are then in that bound's unit, and the fractions at the maximum and at
    the launches' own SM clock follow from the issue-rate probe."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads as wl
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "sm_max_mhz": 2000.0}
    probe = {"flop_per_clk_per_sm": 8192.0}
    w = wl.WORKLOADS["gemm_4096_bf16"]
    ms = w.flops / 1.5e15 * 1e3                       # 1500 TFLOP/s
    r = bench.roofline(w, 1500.0, ms, peaks, "measured", probe, 152, {"sm_mhz_median": 1800.0})
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["frac"] - 0.75) < 1e-12
    assert abs(r["peak_clock_tflops"] - 8192 * 152 * 2000 / 1e6) < 1e-6
    assert abs(r["frac_kernel_clock"] - 1500.0 / (8192 * 152 * 1800 / 1e6)) < 1e-12
    # 256^3: 0.5 MB of compulsory bytes outweigh 34 MFLOP at this peak
    w1 = wl.WORKLOADS["gemm_256_f32out"]
    r1 = bench.roofline(w1, 4.0, w1.flops / 4e12 * 1e3, peaks, "measured", None, 152, None)
    assert r1["bound"] == "hbm" and r1["unit"] == "GB/s"
    assert abs(r1["achieved"] - w1.compulsory_bytes / (w1.flops / 4e12) / 1e9) < 1e-6
    assert "frac_peak_clock" not in r1
    # 8-bit operands: twice the bf16 peak
    w8 = wl.WORKLOADS["gemm_4096_e4m3"]
    assert bench.roofline(w8, 3000.0, 1.0, peaks, "measured", None, 152, None)["peak"] == 4000.0


def test_kernel_clock_summary():
    sys.path.insert(0, ROOT)
    import bench
    rec = [(1800 * 50, 50_000), (1900 * 60, 60_000), (1700 * 70, 70_000), (5, 0)]
    k = bench.kernel_clock(rec)
    assert k["launches"] == 3 and abs(k["sm_mhz_median"] - 1800.0) < 1e-9
    assert abs(k["sm_mhz_min"] - 1700.0) < 1e-9 and abs(k["sm_mhz_max"] - 1900.0) < 1e-9
    assert bench.kernel_clock([]) is None
