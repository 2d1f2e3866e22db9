"""Randomised parity sweep over the plan options and entry points.

Each case draws, from a fixed seed, a shape (ragged M, N, K within the
pitch rules), an operand type, an output type, a unit size, a tile width,
a schedule (static, stream-K, a dynamic work list), a raster group, a CTA
cap, an operand storage (K-major or MN-major) and a batch count, and runs
C = A·Bᵀ through the C ABI on integer inputs in [-4, 4].  Every such sum is
exact in fp32, so the result must equal the fp64 oracle's (rounded once to
a 16-bit output type where one is asked for) element for element; C is
NaN-poisoned first, including a gap between batch elements that must stay
untouched.
"""
from __future__ import annotations

import random

import pytest
import torch

import oracle
import workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu

CASES = 400


def make_case(i: int) -> dict:
    rng = random.Random(20261202 + i)
    dtype = rng.choice([wl.BF16, wl.F16, wl.BF16, wl.F16, wl.E4M3, wl.E5M2])
    fp8 = dtype in wl.FP8
    out = rng.choice([wl.F32, wl.BF16, wl.F16])
    layout = 0 if fp8 else rng.choice([0, 0, 1, 2, 3])
    unit = rng.choice([1, 2, 4])
    K = rng.randrange(1, 80) * (16 if fp8 else 8)
    M = rng.randrange(1, 1600)
    if layout & 1:
        M = -(-M // 8) * 8
    N = rng.randrange(1, 200) * 8
    tile_n = rng.choice([0, 0, 256, 224, 192, 160, 128])
    if layout & 2 and unit == 4:
        tile_n = 0          # the 4-CTA unit holds MN-major B only in whole boxes: let the library pick
    return {"dtype": dtype, "out": out, "layout": layout, "unit": unit, "M": M, "N": N, "K": K,
            "tile_n": tile_n, "dynamic": rng.choice([-1, 0, 1, 2]), "stream_k": rng.choice([0, 0, 1]),
            "group": rng.choice([0, 1, 3, 8]), "cap": rng.choice([0, 0, 0, 8, 24]),
            "batch": rng.choice([1, 1, 1, 3]), "seed": 1000 + i}


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_gemm_blackwell_persistent_gb300 as g
    torch.cuda.set_device(0)
    return g


@pytest.mark.parametrize("i", range(CASES))
def test_random_case_exact(g, i):
    c = make_case(i)
    M, N, K, batch, layout = c["M"], c["N"], c["K"], c["batch"], c["layout"]
    w = wl.Workload("fuzz", M * batch, N * batch, K, c["dtype"], c["out"], "int", c["seed"], lo=-4, hi=4)
    A_all, B_all = wl.make_inputs(w)
    As = [A_all[e * M:(e + 1) * M] for e in range(batch)]
    Bs = [B_all[e * N:(e + 1) * N] for e in range(batch)]

    if c["unit"] == 4 and torch.cuda.device_count() > 1:
        pytest.skip("the library multicasts only while one GPU is visible")
    plan = g.gemm_plan_create(0)
    try:
        g.gemm_plan_set_option(plan, g.GEMM_OPT_CTA_PAIR, 1 if c["unit"] == 1 else 2)
        g.gemm_plan_set_option(plan, g.GEMM_OPT_MULTICAST, 1 if c["unit"] == 4 else 0)
        g.gemm_plan_set_option(plan, g.GEMM_OPT_TILE_N, c["tile_n"])
        g.gemm_plan_set_option(plan, g.GEMM_OPT_DYNAMIC, c["dynamic"])
        g.gemm_plan_set_option(plan, g.GEMM_OPT_STREAM_K, c["stream_k"])
        g.gemm_plan_set_option(plan, g.GEMM_OPT_GROUP_M, c["group"])
        g.gemm_plan_set_option(plan, g.GEMM_OPT_MAX_CTAS, c["cap"])

        # device storage: each element in its layout's storage, elements `pad` apart
        pad = 64

        def stage(mats, mn):
            mats = [m.t().contiguous() if mn else m.contiguous() for m in mats]
            n = mats[0].numel()
            buf = torch.zeros(batch * (n + pad), dtype=mats[0].dtype)
            for e, m in enumerate(mats):
                buf[e * (n + pad):e * (n + pad) + n] = m.reshape(-1)
            return buf.cuda(), n + pad

        Ad, sa = stage(As, layout & 1)
        Bd, sb = stage(Bs, layout & 2)
        sc = M * N + pad
        C = torch.full((batch * sc,), float("nan"), dtype=wl.TORCH_DTYPES[c["out"]], device="cuda")
        stream = torch.cuda.current_stream().cuda_stream
        if batch == 1 and layout == 0:
            g.gemm_plan_run(plan, Ad.data_ptr(), Bd.data_ptr(), C.data_ptr(), M, N, K, c["dtype"], c["out"], stream)
        elif batch == 1:
            g.gemm_plan_run_layout(plan, Ad.data_ptr(), Bd.data_ptr(), C.data_ptr(), M, N, K, c["dtype"], c["out"],
                                   layout, stream)
        else:
            g.gemm_plan_run_batched(plan, Ad.data_ptr(), Bd.data_ptr(), C.data_ptr(), batch, M, N, K, sa, sb, sc,
                                    c["dtype"], c["out"], layout, stream)
        torch.cuda.synchronize()
        assert g.gemm_plan_status(plan) == 0, c
        launch = g.gemm_plan_last_launch(plan)
    finally:
        torch.cuda.synchronize()
        g.gemm_plan_destroy(plan)

    Cv = C.view(batch, sc)
    assert bool(torch.isnan(Cv[:, M * N:].float()).all()), f"padding between outputs was written: {c}"
    for e in range(batch):
        C_ref, _ = oracle.gemm(wl.as_bits(As[e].contiguous()), wl.as_bits(Bs[e].contiguous()), c["dtype"])
        want = C_ref if c["out"] == wl.F32 else oracle.decode(oracle.encode(C_ref, c["out"]), c["out"])
        got = parity.to_f64(Cv[e, :M * N].view(M, N))
        bad = int((got != want).sum())
        assert bad == 0, f"{bad} mismatches in element {e}: {c} launch {launch}"
