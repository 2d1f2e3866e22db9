"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Every test here needs a GB300 and is marked ``gpu``.  Inputs come from the
seeded generators in workloads.py; expected values come only from oracle/.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu

OUTS = [wl.F32, wl.BF16, wl.F16]
FP8S = [wl.E4M3, wl.E5M2]
TORCH = wl.TORCH_DTYPES
CODE_OF = {t: code for code, t in wl.TORCH_DTYPES.items()}


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_gemm_blackwell_persistent_gb300 as g
    return g


@pytest.fixture(scope="module")
def plan(g):
    torch.cuda.set_device(0)
    h = g.gemm_plan_create(0)
    yield h
    torch.cuda.synchronize()
    g.gemm_plan_destroy(h)


@pytest.fixture
def fresh_plan(g):
    torch.cuda.set_device(0)
    h = g.gemm_plan_create(0)
    yield h
    torch.cuda.synchronize()
    g.gemm_plan_destroy(h)


UNITS = [4, 2, 1]   # CTAs per work unit: multicast cluster of two pairs, one pair, one CTA


def configure(g, plan, unit):
    if unit == 4 and torch.cuda.device_count() > 1:
        pytest.skip("the library multicasts only while one GPU is visible")
    g.gemm_plan_set_option(plan, g.GEMM_OPT_CTA_PAIR, 1 if unit == 1 else 2)
    g.gemm_plan_set_option(plan, g.GEMM_OPT_MULTICAST, 1 if unit == 4 else 0)


def run(g, plan, A, B, out_dtype, C=None):
    """C = A·Bᵀ through gemm_plan_run; C is poisoned with NaN first."""
    M, K = A.shape
    N = B.shape[0]
    if C is None:
        C = torch.full((M, N), float("nan"), dtype=TORCH[out_dtype], device="cuda")
    code = CODE_OF[A.dtype]
    g.gemm_plan_run(plan, A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, code, out_dtype,
                    torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert g.gemm_plan_status(plan) == 0
    return C


def oracle_full(A, B):
    return oracle.gemm(wl.as_bits(A), wl.as_bits(B), CODE_OF[A.dtype])


def draw(M, N, K, dtype=wl.BF16, dist="normal", seed=0):
    w = wl.Workload("case", M, N, K, dtype, wl.F32, dist, seed,
                    lo=-4 if dist == "int" else -1.0, hi=4 if dist == "int" else 1.0)
    return wl.make_inputs(w)


# ------------------------------------------------------------------ bit-exact integer runs

@pytest.mark.parametrize("unit", UNITS)
@pytest.mark.parametrize("out", OUTS)
@pytest.mark.parametrize("shape", [(256, 256, 256), (200, 136, 264), (384, 512, 1024), (1100, 520, 136)])
def test_integer_inputs_bit_exact(g, plan, unit, out, shape):
    M, N, K = shape
    configure(g, plan, unit)
    try:
        A, B = draw(M, N, K, dist="int", seed=0)
        C = parity.to_f64(run(g, plan, A.cuda(), B.cuda(), out))
        C_ref, _ = oracle_full(A, B)
        if out == wl.F32:
            want = C_ref
        else:
            want = oracle.decode(oracle.encode(C_ref, out), out)
        assert np.array_equal(C, want), f"{int((C != want).sum())} mismatches"
    finally:
        configure(g, plan, 4)


def test_integer_workload_256(g, plan):
    w = wl.WORKLOADS["gemm_256_int"]
    A, B = wl.make_inputs(w)
    C = parity.to_f64(run(g, plan, A.cuda(), B.cuda(), w.out_dtype))
    C_ref, _ = oracle_full(A, B)
    assert np.array_equal(C, C_ref)


# ------------------------------------------------------------------ random inputs, full comparison

def test_workload_256_f32out(g, plan):
    w = wl.WORKLOADS["gemm_256_f32out"]
    A, B = wl.make_inputs(w)
    C = parity.to_f64(run(g, plan, A.cuda(), B.cuda(), w.out_dtype))
    C_ref, S = oracle_full(A, B)
    parity.assert_within(C, C_ref, S, w.out_dtype, w.name)


SHAPES = [
    (8, 8, 8), (1, 8, 16), (3, 16, 24), (128, 256, 64), (129, 264, 72), (255, 248, 136),
    (256, 256, 128), (257, 264, 200), (384, 520, 1000), (1000, 776, 520), (640, 1288, 64),
]


@pytest.mark.parametrize("unit", UNITS)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_shape_sweep(g, plan, unit, shape):
    M, N, K = shape
    configure(g, plan, unit)
    try:
        for i, out in enumerate(OUTS):
            dtype = wl.BF16 if (i + M) % 2 == 0 else wl.F16
            A, B = draw(M, N, K, dtype=dtype, seed=M * 7 + N * 3 + K + i)
            C = parity.to_f64(run(g, plan, A.cuda(), B.cuda(), out))
            C_ref, S = oracle_full(A, B)
            parity.assert_within(C, C_ref, S, out, f"{shape} unit={unit} out={out} in={dtype}")
    finally:
        configure(g, plan, 4)


@pytest.mark.parametrize("unit,ctas,group", [(2, 2, 8), (2, 6, 3), (1, 1, 8), (1, 5, 1), (2, 4, 1),
                                             (4, 4, 8), (4, 8, 1), (4, 12, 2)])
def test_persistent_loop_many_tiles(g, fresh_plan, unit, ctas, group):
    """Few resident CTAs, many tiles each: wraps the shared-memory ring many
    times and alternates both TMEM accumulators across tiles."""
    configure(g, fresh_plan, unit)
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_MAX_CTAS, ctas)
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_GROUP_M, group)
    M, N, K = 1100, 1288, 328
    for out in OUTS:
        A, B = draw(M, N, K, seed=ctas * 10 + group + out)
        C = parity.to_f64(run(g, fresh_plan, A.cuda(), B.cuda(), out))
        assert g.gemm_plan_last_grid(fresh_plan) == ctas // unit * unit
        C_ref, S = oracle_full(A, B)
        parity.assert_within(C, C_ref, S, out, f"unit={unit} ctas={ctas} group={group} out={out}")


TILE_NS = [256, 224, 192, 160, 128]



@pytest.mark.parametrize("unit", UNITS)
@pytest.mark.parametrize("tile_n", TILE_NS)
def test_every_tile_width(g, fresh_plan, unit, tile_n):
    """Each instantiated tile width, every unit size, all output types: ragged
    in M, N and K, several tiles in each direction, few CTAs so each walks
    many tiles; integer inputs bit-exact, random inputs within tolerance."""
    configure(g, fresh_plan, unit)
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_TILE_N, tile_n)
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_MAX_CTAS, 8)
    pair = unit
    M, N, K = 600, 1000, 392
    for out in OUTS:
        A, B = draw(M, N, K, dist="int", seed=tile_n + out)
        C = parity.to_f64(run(g, fresh_plan, A.cuda(), B.cuda(), out))
        assert g.gemm_plan_last_tile_n(fresh_plan) == tile_n
        C_ref, _ = oracle_full(A, B)
        want = C_ref if out == wl.F32 else oracle.decode(oracle.encode(C_ref, out), out)
        assert np.array_equal(C, want), f"tile_n={tile_n} pair={pair} out={out}"
        dtype = wl.F16 if out == wl.F16 else wl.BF16
        A, B = draw(M, N, K, dtype=dtype, seed=tile_n * 3 + out)
        C = parity.to_f64(run(g, fresh_plan, A.cuda(), B.cuda(), out))
        C_ref, S = oracle_full(A, B)
        parity.assert_within(C, C_ref, S, out, f"tile_n={tile_n} pair={pair} out={out}")


@pytest.mark.parametrize("name,expect", [("gemm_4096_bf16", (224, 152, 4)),
                                         ("gemm_1024x4096x4096_f16", (224, 152, 1)),
                                         ("gemm_8192_bf16", (256, 224, 13))])
def test_default_launch_of_workloads(g, fresh_plan, name, expect):
    """Tile width: the candidate with the fewest waves × measured cycles per
    k-block, so a narrower tile where it turns a partial last wave into
    whole waves.  Schedule: static where the tiles fill whole waves (4096³:
    304 tiles = 4 waves on 76 pairs); at 8192³ (1024 tiles = 13 waves + 36)
    the 76 persistent pairs keep 13 waves each and the 36 tiles of the
    partial wave are handed out at run time (76 + 36 clusters of 2 CTAs)."""
    w = wl.WORKLOADS[name]
    A = torch.zeros((w.M, w.K), dtype=wl.TORCH_DTYPES[w.dtype], device="cuda")
    B = torch.zeros((w.N, w.K), dtype=wl.TORCH_DTYPES[w.dtype], device="cuda")
    C = run(g, fresh_plan, A, B, w.out_dtype)
    assert bool((C == 0).all())
    launch = g.gemm_plan_last_launch(fresh_plan)
    assert launch["ctas_per_unit"] == 2, launch
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert (launch["tile_n"], launch["ctas"], launch["dp_waves"]) == expect, launch


# (M, N, K, tile width, {CTAs per unit: CTA cap}): shapes whose schedule
# splits tiles along K, for every unit size
STREAM_K_CASES = [
    # fewer tiles than half the units: every tile halved along K
    (1024, 1280, 2048, 256, {1: 0, 2: 0, 4: 0}),
    # a partial last wave: the last whole wave and the rest spread over all units
    (1300, 1096, 2000, 256, {1: 16, 2: 14, 4: 8}),
    # the same, ragged M/N and a partial last k-block
    (520, 776, 2056, 128, {1: 8, 2: 8, 4: 16}),
]


@pytest.mark.parametrize("unit", UNITS)
@pytest.mark.parametrize("case", STREAM_K_CASES, ids=lambda c: "x".join(map(str, c[:3])))
def test_stream_k(g, fresh_plan, unit, case):
    M, N, K, tile_n, caps = case
    configure(g, fresh_plan, unit)
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_MAX_CTAS, caps[unit])
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_TILE_N, tile_n)
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_STREAM_K, 1)
    for out in OUTS:
        # integer inputs: exact whatever the split
        A, B = draw(M, N, K, dist="int", seed=K + out)
        C = parity.to_f64(run(g, fresh_plan, A.cuda(), B.cuda(), out))
        assert g.gemm_plan_last_launch(fresh_plan)["sk_tiles"] > 0, "the schedule did not split"
        C_ref, _ = oracle_full(A, B)
        want = C_ref if out == wl.F32 else oracle.decode(oracle.encode(C_ref, out), out)
        assert np.array_equal(C, want), f"stream-K {case} unit={unit} out={out}"
        # random inputs: tolerance, and bitwise repeatable
        dtype = wl.F16 if out == wl.F16 else wl.BF16
        A, B = draw(M, N, K, dtype=dtype, seed=K * 7 + out)
        Ad, Bd = A.cuda(), B.cuda()
        C1 = run(g, fresh_plan, Ad, Bd, out)
        C2 = run(g, fresh_plan, Ad, Bd, out)
        assert torch.equal(C1.view(torch.uint8), C2.view(torch.uint8)), "stream-K result not repeatable"
        C_ref, S = oracle_full(A, B)
        parity.assert_within(parity.to_f64(C1), C_ref, S, out, f"stream-K {case} unit={unit} out={out}")


def test_stream_k_off_matches_within_tolerance(g, fresh_plan):
    M, N, K = 1024, 1280, 1024
    A, B = draw(M, N, K, seed=77)
    Ad, Bd = A.cuda(), B.cuda()
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_STREAM_K, 1)
    C_on = parity.to_f64(run(g, fresh_plan, Ad, Bd, wl.F32))
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_STREAM_K, 0)
    C_off = parity.to_f64(run(g, fresh_plan, Ad, Bd, wl.F32))
    C_ref, S = oracle_full(A, B)
    parity.assert_within(C_on, C_ref, S, wl.F32, "stream-K on")
    parity.assert_within(C_off, C_ref, S, wl.F32, "stream-K off")


# ------------------------------------------------------------------ dynamic tile scheduling

# (M, N, K, tile width): several tiles per resident unit, ragged edges and a
# partial last k-block; one-k-block tiles, so that units come back for work
# quickly and the response ring wraps many times.  With every resident unit
# (152 CTAs as singles or pairs, 144 in 4-CTA clusters) the tile counts leave
# a partial last wave, and the first case fits in one wave.
DYNAMIC_CASES = [
    (1300, 1096, 520, 224),
    (2048, 2048, 264, 128),
    (4096, 4096, 64, 128),
]


def tiles_of(M, N, unit, tile_n, batch=1):
    return batch * (-(-M // (128 * unit))) * (-(-N // tile_n))


@pytest.mark.parametrize("mode", [1, 2], ids=["tail", "every_tile"])
@pytest.mark.parametrize("unit", UNITS)
@pytest.mark.parametrize("case", DYNAMIC_CASES, ids=lambda c: "x".join(map(str, c[:3])))
def test_dynamic_schedule(g, fresh_plan, unit, case, mode):
    """Clusters that finish their list of tiles take over the lists of
    clusters that have not started (cluster launch control).  Every tile
    must be computed exactly once: integer inputs give the oracle's exact
    sums."""
    M, N, K, tile_n = case
    configure(g, fresh_plan, unit)
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_TILE_N, tile_n)
    T = tiles_of(M, N, unit, tile_n)
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_DYNAMIC, 0)
    A, B = draw(M, N, K, dist="int", seed=K + 2)
    C_ref, _ = oracle_full(A, B)
    Ad, Bd = A.cuda(), B.cuda()
    run(g, fresh_plan, Ad, Bd, wl.F32)
    static = g.gemm_plan_last_launch(fresh_plan)
    P = static["ctas"] // unit   # resident units (or the tiles, if fewer)
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_DYNAMIC, mode)
    for out in OUTS:
        C = parity.to_f64(run(g, fresh_plan, Ad, Bd, out))
        launch = g.gemm_plan_last_launch(fresh_plan)
        if mode == 2:
            assert (launch["ctas"], launch["dp_waves"]) == (T * unit, 0), launch
        elif T > P and T % P:
            assert (launch["ctas"], launch["dp_waves"]) == ((P + T % P) * unit, T // P), (launch, T, P)
        else:
            assert launch == static, (launch, static)
        want = C_ref if out == wl.F32 else oracle.decode(oracle.encode(C_ref, out), out)
        assert np.array_equal(C, want), f"dynamic {case} unit={unit} out={out}: {int((C != want).sum())} mismatches"
    A, B = draw(M, N, K, dtype=wl.BF16, seed=K * 5 + 1)
    C_ref, S = oracle_full(A, B)
    parity.assert_within(parity.to_f64(run(g, fresh_plan, A.cuda(), B.cuda(), wl.BF16)), C_ref, S, wl.BF16,
                         f"dynamic {case} unit={unit}")


@pytest.mark.parametrize("unit", UNITS)
def test_dynamic_batched_and_fp8(g, fresh_plan, unit):
    configure(g, fresh_plan, unit)
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_DYNAMIC, 2)
    case = (5, 520, 776, 1008, False, False, 0, 0)
    As, Bs = draw_batch(case, "int", seed=40 + unit)
    Cs = run_batched(g, fresh_plan, As, Bs, case, wl.F32)
    assert g.gemm_plan_last_launch(fresh_plan)["dp_waves"] == 0
    for e in range(case[0]):
        C_ref, _ = oracle_full(As[e].contiguous(), Bs[e].contiguous())
        assert np.array_equal(parity.to_f64(Cs[e]), C_ref), f"batch element {e}"
    A, B = draw(1100, 1096, 1024, dtype=wl.E4M3, dist="int", seed=41)
    C = parity.to_f64(run(g, fresh_plan, A.cuda(), B.cuda(), wl.F32))
    C_ref, _ = oracle_full(A, B)
    assert np.array_equal(C, C_ref)


def test_dynamic_by_default_on_many_waves(g, fresh_plan):
    """With default options, a product of 6 or more whole waves and a
    partial one hands the partial wave out at run time: here 32 batched
    1024×1024×128 products, 512 tiles of 256×256 on 76 pairs = 6 waves + 56
    tiles, so 76 + 56 clusters.  Every element exact for integer inputs."""
    case = (32, 1024, 1024, 128, False, False, 0, 0)
    As, Bs = draw_batch(case, "int", seed=45)
    Cs = run_batched(g, fresh_plan, As, Bs, case, wl.F32)
    launch = g.gemm_plan_last_launch(fresh_plan)
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert (launch["ctas"], launch["tile_n"], launch["dp_waves"]) == ((76 + 56) * 2, 256, 6), launch
    for e in range(case[0]):
        C_ref, _ = oracle_full(As[e].contiguous(), Bs[e].contiguous())
        assert np.array_equal(parity.to_f64(Cs[e]), C_ref), f"batch element {e}"


@pytest.mark.parametrize("mode", [1, 2], ids=["tail", "every_tile"])
def test_dynamic_schedule_in_cuda_graph(g, fresh_plan, mode):
    """A run with a dynamic work list recorded into a CUDA graph: each replay
    launches the grid again and the running clusters cancel the ones that
    have not started, so every replay must compute every tile once.
    2048×4096×64 with 256×128 pair tiles is 256 tiles (3 waves + 28 on 76
    pairs: 104 or 256 clusters launched); replays on new integer inputs must
    equal the oracle exactly."""
    M, N, K = 2048, 4096, 64
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_TILE_N, 128)
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_DYNAMIC, mode)
    Ad = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    Bd = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    Cd = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g.gemm_plan_run(fresh_plan, Ad.data_ptr(), Bd.data_ptr(), Cd.data_ptr(), M, N, K, wl.BF16, wl.F32,
                        s.cuda_stream)
    s.synchronize()
    assert g.gemm_plan_last_launch(fresh_plan)["ctas"] > 152 or \
        torch.cuda.get_device_properties(0).multi_processor_count != 152
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        g.gemm_plan_run(fresh_plan, Ad.data_ptr(), Bd.data_ptr(), Cd.data_ptr(), M, N, K, wl.BF16, wl.F32,
                        torch.cuda.current_stream().cuda_stream)
    for seed in (51, 52):
        A, B = draw(M, N, K, dist="int", seed=seed)
        Ad.copy_(A)
        Bd.copy_(B)
        Cd.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert g.gemm_plan_status(fresh_plan) == 0
        C_ref, _ = oracle_full(A, B)
        assert np.array_equal(parity.to_f64(Cd), C_ref), f"replay with seed {seed}"


def test_many_launches_mixed_schedules(g):
    """Back-to-back launches cycling through every schedule (static, stream-K,
    dynamic work lists) and unit size on two streams at once, each plan kept
    on one stream: every result stays exact.  Catches state that leaks from
    one launch into the next (stream-K flags, response rings, accumulators)."""
    shapes = [(2048, 4096, 64), (1300, 1096, 520), (768, 3072, 264)]
    data = []
    for i, (M, N, K) in enumerate(shapes):
        A, B = draw(M, N, K, dist="int", seed=900 + i)
        C_ref, _ = oracle_full(A, B)
        data.append((M, N, K, A.cuda(), B.cuda(), torch.from_numpy(C_ref)))
    configs = [(d, sk, u) for d in (0, 1, 2) for sk in (0, 1) for u in UNITS]
    plans = []
    for d, sk, u in configs:
        p = g.gemm_plan_create(0)
        configure(g, p, u)
        g.gemm_plan_set_option(p, g.GEMM_OPT_DYNAMIC, d)
        g.gemm_plan_set_option(p, g.GEMM_OPT_STREAM_K, sk)
        plans.append(p)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    try:
        pending = []
        for it in range(20 * len(configs)):
            si, ci = it % len(shapes), (it // len(shapes)) % len(configs)
            M, N, K, Ad, Bd, _ = data[si]
            st = streams[ci % 2]
            C = torch.full((M, N), float("nan"), device="cuda")
            with torch.cuda.stream(st):
                g.gemm_plan_run(plans[ci], Ad.data_ptr(), Bd.data_ptr(), C.data_ptr(), M, N, K, wl.BF16, wl.F32,
                                st.cuda_stream)
            pending.append((it, C, si))
            if len(pending) == 24:
                torch.cuda.synchronize()
                for j, Cj, sj in pending:
                    cfg = configs[(j // len(shapes)) % len(configs)]
                    assert torch.equal(Cj.cpu().double(), data[sj][5]), f"launch {j}: {shapes[sj]} {cfg}"
                pending.clear()
        torch.cuda.synchronize()
        for j, Cj, sj in pending:
            assert torch.equal(Cj.cpu().double(), data[sj][5]), f"launch {j}"
        for p in plans:
            assert g.gemm_plan_status(p) == 0
    finally:
        torch.cuda.synchronize()
        for p in plans:
            g.gemm_plan_destroy(p)


def test_host_threads_share_one_plan(g, fresh_plan):
    """Four host threads, each on a stream of its own, run products of their
    own shapes through one plan at the same time (the C calls release the
    GIL, so the library's host code runs concurrently too): every result is
    exact, the last-launch record stays readable throughout, and the plan's
    device status stays clean."""
    import threading
    shapes = [(1300, 1096, 520), (768, 3072, 264), (2048, 1024, 136), (520, 776, 1032)]
    data = []
    for i, (M, N, K) in enumerate(shapes):
        A, B = draw(M, N, K, dist="int", seed=950 + i)
        C_ref, _ = oracle_full(A, B)
        data.append((A.cuda(), B.cuda(), torch.from_numpy(C_ref)))
    torch.cuda.synchronize()
    errors = []
    start = threading.Barrier(len(shapes))

    def worker(t):
        try:
            torch.cuda.set_device(0)
            M, N, K = shapes[t]
            Ad, Bd, C_ref = data[t]
            st = torch.cuda.Stream()
            outs = []
            start.wait()
            with torch.cuda.stream(st):
                for _ in range(30):
                    C = torch.full((M, N), float("nan"), device="cuda")
                    g.gemm_plan_run(fresh_plan, Ad.data_ptr(), Bd.data_ptr(), C.data_ptr(), M, N, K, wl.BF16,
                                    wl.F32, st.cuda_stream)
                    launch = g.gemm_plan_last_launch(fresh_plan)
                    assert launch["ctas_per_unit"] in (1, 2, 4) and launch["ctas"] > 0, launch
                    outs.append(C)
            st.synchronize()
            for j, C in enumerate(outs):
                if not torch.equal(C.cpu().double(), C_ref):
                    errors.append(f"thread {t}, launch {j}: {shapes[t]} not exact")
                    break
        except Exception as e:   # reported below: an exception in a thread would be lost
            errors.append(f"thread {t}: {e!r}")

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(len(shapes))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    assert not errors, errors
    assert g.gemm_plan_status(fresh_plan) == 0


def test_multicast_only_with_one_visible_gpu(g, fresh_plan):
    """TMA multicast stays within one GPU's memory and the library uses it
    only while the process sees a single GPU.  Rows of 1256 bf16 (2512
    bytes, not a multiple of 128) make the default pick the 4-CTA multicast
    unit with one GPU visible; counted as two, the same plan picks pairs
    and refuses an explicit multicast request.  Results exact either way.
    Skipped where the process sees more than one GPU: there the library's
    own guard must not be overridden."""
    if torch.cuda.device_count() > 1:
        pytest.skip("the library multicasts only while one GPU is visible")
    M, N, K = 1000, 776, 1256
    A, B = draw(M, N, K, dist="int", seed=77)
    C_ref, _ = oracle_full(A, B)
    Ad, Bd = A.cuda(), B.cuda()
    opt = g.GEMM_OPT_VISIBLE_DEVICES
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_CTA_PAIR, 2)   # pairs: this product is small enough for single CTAs
    try:
        for visible, unit in ((1, 4), (2, 2)):
            g.gemm_plan_set_option(fresh_plan, opt, visible)
            C = parity.to_f64(run(g, fresh_plan, Ad, Bd, wl.F32))
            assert g.gemm_plan_last_launch(fresh_plan)["ctas_per_unit"] == unit, visible
            assert np.array_equal(C, C_ref), visible
        g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_MULTICAST, 1)
        C = torch.full((M, N), float("nan"), device="cuda")
        import ctypes
        vp = ctypes.c_void_p
        assert g.raw_status("gemm_plan_run", vp(fresh_plan), vp(Ad.data_ptr()), vp(Bd.data_ptr()), vp(C.data_ptr()),
                            M, N, K, wl.BF16, wl.F32, None) == g.GEMM_ERR_UNSUPPORTED
        torch.cuda.synchronize()
        assert bool(torch.isnan(C).all()), "a refused run wrote C"
        g.gemm_plan_set_option(fresh_plan, opt, 1)
        C = parity.to_f64(run(g, fresh_plan, Ad, Bd, wl.F32))
        assert g.gemm_plan_last_launch(fresh_plan)["ctas_per_unit"] == 4
        assert np.array_equal(C, C_ref)
    finally:
        g.gemm_plan_set_option(fresh_plan, opt, 0)
        g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_MULTICAST, -1)
    for bad in (-1, 1025):
        import ctypes
        assert g.raw_status("gemm_plan_set_option", ctypes.c_void_p(fresh_plan), opt, ctypes.c_int64(bad)) \
            == g.GEMM_ERR_INVALID_ARG


def test_dynamic_and_static_agree(g, fresh_plan):
    """The schedule decides only where a tile is computed, not how: the
    same inputs give bitwise the same C every way."""
    M, N, K = 3000, 2800, 1000
    A, B = draw(M, N, K, seed=43)
    Ad, Bd = A.cuda(), B.cuda()
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_DYNAMIC, 0)
    C_sta = run(g, fresh_plan, Ad, Bd, wl.F32)
    for mode in (1, 2):
        g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_DYNAMIC, mode)
        C_dyn = run(g, fresh_plan, Ad, Bd, wl.F32)
        assert torch.equal(C_dyn, C_sta), f"mode {mode}"
    C_ref, S = oracle_full(A, B)
    parity.assert_within(parity.to_f64(C_dyn), C_ref, S, wl.F32, "dynamic")


# ------------------------------------------------------------------ tensor-core issue-rate probe

@pytest.mark.parametrize("dtype,nominal", [(wl.BF16, 8192), (wl.F16, 8192), (wl.E4M3, 16384), (wl.E5M2, 16384)],
                         ids=["bf16", "f16", "e4m3", "e5m2"])
@pytest.mark.parametrize("pair", [2, 1])
def test_mma_probe_rate(g, dtype, nominal, pair):
    """Back-to-back MMAs with no loads run at the tensor cores' dense rate:
    8192 FLOP per SM clock for 16-bit operands and twice that for 8-bit
    ones (NVIDIA's dense figures divided by SMs × clock), and the all-SM
    rate agrees with that rate × SMs × the clock measured alongside."""
    r = g.gemm_probe_mma_rate(dtype, pair, 1 << 16)
    assert abs(r["flop_per_clk_per_sm"] / nominal - 1) < 0.02, r
    assert 300 < r["sm_mhz"] < 2200, r
    sms = torch.cuda.get_device_properties(0).multi_processor_count // pair * pair
    expect = r["flop_per_clk_per_sm"] * sms * r["sm_mhz"] * 1e6 / 1e12
    assert 0.8 < r["tflops"] / expect < 1.1, (r, expect)


@pytest.mark.parametrize("tile_n", [256, 224, 192, 160, 128, 64])
def test_mma_probe_rate_by_tile_width(g, tile_n):
    """The tensor cores' own rate for a pair's 256×N instructions: the full
    dense rate at every GEMM tile width from 128 to 256 (so a narrow tile
    that runs slower per k-block than its MMA work is held up by feeding,
    not by the MMA); N = 64 is below it (measured ~5660 FLOP/clk/SM)."""
    r = g.gemm_probe_mma_rate(wl.BF16, 2, 1 << 15, tile_n=tile_n)
    if tile_n >= 128:
        assert abs(r["flop_per_clk_per_sm"] / 8192 - 1) < 0.02, r
    else:
        assert 0 < r["flop_per_clk_per_sm"] < 8192 * 1.02, r


def test_mma_probe_arguments(g):
    import ctypes
    d = ctypes.c_double()
    for args in ((wl.F32, 2, 1 << 12), (wl.BF16, 3, 1 << 12), (wl.BF16, 2, 6), (wl.BF16, 2, 0), (wl.BF16, 2, 1 << 25)):
        assert g.raw_status("gemm_probe_mma_rate", *args, ctypes.byref(d), None, None) == g.GEMM_ERR_INVALID_ARG
    for n in (0, 8, 100, 272):
        assert g.raw_status("gemm_probe_mma_rate_n", wl.BF16, 2, n, 1 << 12, ctypes.byref(d), None, None) \
            == g.GEMM_ERR_INVALID_ARG


# ------------------------------------------------------------------ 8-bit float inputs

@pytest.mark.parametrize("unit", UNITS)
@pytest.mark.parametrize("fp8", FP8S, ids=["e4m3", "e5m2"])
@pytest.mark.parametrize("out", OUTS)
@pytest.mark.parametrize("shape", [(256, 256, 256), (200, 136, 272), (384, 512, 1024), (1100, 520, 144)])
def test_fp8_integer_inputs_bit_exact(g, plan, unit, fp8, out, shape):
    """Integers -4..4 are exact in both 8-bit formats and every partial sum is
    exact in fp32: any correct kernel gives the oracle's bits.  K = 272 and
    144 end in a partial 128-element k-block (zero-filled by TMA)."""
    M, N, K = shape
    configure(g, plan, unit)
    try:
        w = wl.Workload("case", M, N, K, fp8, out, "int", 40 + K, lo=-4, hi=4)
        A, B = wl.make_inputs(w)
        C = parity.to_f64(run(g, plan, A.cuda(), B.cuda(), out))
        C_ref, _ = oracle_full(A, B)
        want = C_ref if out == wl.F32 else oracle.decode(oracle.encode(C_ref, out), out)
        assert np.array_equal(C, want), f"{int((C != want).sum())} mismatches"
    finally:
        configure(g, plan, 4)


@pytest.mark.parametrize("unit", UNITS)
@pytest.mark.parametrize("fp8", FP8S, ids=["e4m3", "e5m2"])
@pytest.mark.parametrize("shape", [(512, 384, 2048), (1000, 760, 1264)])
def test_fp8_random_within_tolerance(g, plan, unit, fp8, shape):
    M, N, K = shape
    configure(g, plan, unit)
    try:
        w = wl.Workload("case", M, N, K, fp8, wl.F32, "normal", 50 + K)
        A, B = wl.make_inputs(w)
        Ad, Bd = A.cuda(), B.cuda()
        C_ref, S = oracle_full(A, B)
        for out in OUTS:
            C = parity.to_f64(run(g, plan, Ad, Bd, out))
            parity.assert_within(C, C_ref, S, out, f"fp8 {fp8} {shape} unit={unit} out={out}")
    finally:
        configure(g, plan, 4)


def test_fp8_matmul_helper(g, plan):
    w = wl.Workload("case", 300, 264, 400, wl.E4M3, wl.BF16, "int", 61, lo=-4, hi=4)
    A, B = wl.make_inputs(w)
    C = g.matmul(A.cuda(), B.cuda())
    torch.cuda.synchronize()
    assert C.dtype == torch.bfloat16
    C_ref, _ = oracle_full(A, B)
    assert np.array_equal(parity.to_f64(C), oracle.decode(oracle.encode(C_ref, wl.BF16), wl.BF16))


def test_fp8_k_must_fill_16_bytes(g, plan):
    A = torch.zeros((64, 24), dtype=torch.float8_e4m3fn, device="cuda")
    C = torch.zeros((64, 64), dtype=torch.float32, device="cuda")
    import ctypes
    vp = ctypes.c_void_p
    assert g.raw_status("gemm_plan_run", vp(plan), vp(A.data_ptr()), vp(A.data_ptr()), vp(C.data_ptr()),
                        64, 64, 24, g.GEMM_E4M3, g.GEMM_F32, None) == g.GEMM_ERR_UNSUPPORTED


# ------------------------------------------------------------------ operand majors

LAYOUTS = {1: "A_KxM", 2: "B_KxN", 3: "both"}


def run_layout(g, plan, A, B, layout, out_dtype):
    """C = A·Bᵀ with A [M,K], B [N,K] handed over in `layout`'s storage."""
    M, K = A.shape
    N = B.shape[0]
    As = A.t().contiguous() if layout & 1 else A
    Bs = B.t().contiguous() if layout & 2 else B
    C = torch.full((M, N), float("nan"), dtype=TORCH[out_dtype], device="cuda")
    g.gemm_plan_run_layout(plan, As.data_ptr(), Bs.data_ptr(), C.data_ptr(), M, N, K, CODE_OF[A.dtype], out_dtype,
                           layout, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert g.gemm_plan_status(plan) == 0
    return C


@pytest.mark.parametrize("unit", UNITS)
@pytest.mark.parametrize("layout", list(LAYOUTS), ids=list(LAYOUTS.values()))
@pytest.mark.parametrize("shape", [(256, 256, 256), (200, 136, 264), (384, 512, 1024), (1096, 520, 136)])
def test_operand_majors_integer_bit_exact(g, plan, unit, layout, shape):
    """A stored K×M and/or B stored K×N, read in place (MN-major tiles):
    integers give the oracle's bits; ragged M, N and K included."""
    M, N, K = shape
    configure(g, plan, unit)
    try:
        A, B = draw(M, N, K, dist="int", seed=70 + layout)
        C = parity.to_f64(run_layout(g, plan, A.cuda(), B.cuda(), layout, wl.F32))
        C_ref, _ = oracle_full(A, B)
        assert np.array_equal(C, C_ref), f"{int((C != C_ref).sum())} mismatches"
    finally:
        configure(g, plan, 4)


@pytest.mark.parametrize("unit", UNITS)
@pytest.mark.parametrize("layout", list(LAYOUTS), ids=list(LAYOUTS.values()))
def test_operand_majors_random_within_tolerance(g, plan, unit, layout):
    configure(g, plan, unit)
    try:
        for dtype, out in ((wl.BF16, wl.BF16), (wl.F16, wl.F16), (wl.BF16, wl.F32)):
            A, B = draw(1000, 776, 1256, dtype=dtype, seed=80 + layout)
            C = parity.to_f64(run_layout(g, plan, A.cuda(), B.cuda(), layout, out))
            C_ref, S = oracle_full(A, B)
            parity.assert_within(C, C_ref, S, out, f"layout {LAYOUTS[layout]} unit={unit} out={out}")
    finally:
        configure(g, plan, 4)


def test_plain_a_times_b_full_size(g, plan):
    """bf16 4096³ with B a plain row-major K×N matrix (C = A·B), the layout of
    the pages' Pallas matmuls, at full size: every output against the oracle."""
    w = wl.WORKLOADS["gemm_4096_bf16"]
    A, B = wl.make_inputs(w)                     # B drawn N×K; handed over as K×N
    got = parity.to_f64(run_layout(g, plan, A.cuda(), B.cuda(), 2, w.out_dtype))
    C_ref, S = oracle_full(A, B)
    parity.assert_within(got, C_ref, S, w.out_dtype, "A·B, B K×N")


def test_matmul_helper_operand_majors(g, plan):
    A, B = draw(264, 328, 200, seed=91)
    Ad, Bd = A.cuda(), B.cuda()
    C_ref, S = oracle_full(A, B)
    Akm, Bkn = Ad.t().contiguous(), Bd.t().contiguous()
    for kw, a, b in (({"b_kn": True}, Ad, Bkn), ({"a_km": True}, Akm, Bd), ({"a_km": True, "b_kn": True}, Akm, Bkn)):
        C = g.matmul(a, b, out_dtype=torch.float32, plan=plan, **kw)
        torch.cuda.synchronize()
        parity.assert_within(parity.to_f64(C), C_ref, S, wl.F32, str(kw))


def test_operand_major_rules(g, plan):
    import ctypes
    vp = ctypes.c_void_p
    A = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((64, 64), dtype=torch.float32, device="cuda")
    args = (vp(plan), vp(A.data_ptr()), vp(A.data_ptr()), vp(C.data_ptr()))
    rs = g.raw_status
    assert rs("gemm_plan_run_layout", *args, 64, 64, 64, 0, 2, 4, None) == g.GEMM_ERR_INVALID_ARG
    assert rs("gemm_plan_run_layout", *args, 64, 64, 64, 3, 2, 1, None) == g.GEMM_ERR_UNSUPPORTED  # fp8
    assert rs("gemm_plan_run_layout", *args, 60, 64, 64, 0, 2, 1, None) == g.GEMM_ERR_UNSUPPORTED  # M*2 % 16
    assert rs("gemm_plan_run_layout", *args, 64, 64, 60, 0, 2, 3, None) == g.GEMM_OK   # K free when both MN-major
    torch.cuda.synchronize()
    assert g.gemm_plan_status(plan) == 0
    fresh = g.gemm_plan_create(0)
    try:
        # a 4-CTA unit loads a 56-row quarter of a 224-wide B tile: not whole boxes
        g.gemm_plan_set_option(fresh, g.GEMM_OPT_TILE_N, 224)
        g.gemm_plan_set_option(fresh, g.GEMM_OPT_MULTICAST, 1)
        assert rs("gemm_plan_run_layout", vp(fresh), *args[1:], 64, 64, 64, 0, 2, 2, None) == g.GEMM_ERR_UNSUPPORTED
    finally:
        g.gemm_plan_destroy(fresh)


@pytest.mark.parametrize("unit", [2, 1])
@pytest.mark.parametrize("tile_n", TILE_NS)
@pytest.mark.parametrize("layout", [2, 3], ids=["B_KxN", "both"])
def test_operand_major_b_every_tile_width(g, fresh_plan, unit, tile_n, layout):
    """An MN-major B at every tile width; where a CTA's share of B is not whole
    64-element boxes (e.g. 112 rows of a 256×224 pair tile) the padded kernel
    form loads whole boxes and the MMA reads only the share."""
    configure(g, fresh_plan, unit)
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_TILE_N, tile_n)
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_MAX_CTAS, 8)   # several tiles per unit
    M, N, K = 600, 1000, 392
    A, B = draw(M, N, K, dist="int", seed=95 + tile_n)
    C = parity.to_f64(run_layout(g, fresh_plan, A.cuda(), B.cuda(), layout, wl.F32))
    assert g.gemm_plan_last_tile_n(fresh_plan) == tile_n
    C_ref, _ = oracle_full(A, B)
    assert np.array_equal(C, C_ref), f"{int((C != C_ref).sum())} mismatches"


# ------------------------------------------------------------------ batched products

# (batch, M, N, K, A shared, B shared, layout, stride padding in elements)
BATCH_CASES = [
    # the shape of the batched masked matmul of "Chapter 7: Writing Custom
    # Kernels with Pallas", §5.2 (vmap over 3, B K×N shared), with N 130 -> 136
    # so that rows are 16-byte multiples
    (3, 100, 136, 200, False, True, 2, 0),
    (4, 260, 520, 264, False, False, 0, 64),    # separate A and B, padded batch strides
    (5, 256, 264, 136, True, False, 0, 0),      # A shared
    (2, 1000, 776, 392, False, False, 3, 8),    # both operands MN-major
]


def run_batched(g, plan, As, Bs, case, out):
    """As: [batch,M,K] CPU tensors (or one shared [M,K]); Bs likewise [N,K]."""
    batch, M, N, K, a_sh, b_sh, layout, pad = case
    dt = CODE_OF[As.dtype]

    def stage(X, rows, cols, shared, mn):
        # device storage: each element row-major (or its transpose for an MN-major operand), `pad` apart
        mats = [X] if shared else [X[e] for e in range(batch)]
        mats = [m.t().contiguous() if mn else m.contiguous() for m in mats]
        if shared:
            return mats[0].cuda(), 0
        stride = rows * cols + pad
        buf = torch.zeros(batch * stride, dtype=X.dtype)
        for e, m in enumerate(mats):
            buf[e * stride:e * stride + rows * cols] = m.reshape(-1)
        return buf.cuda(), stride

    Ad, sa = stage(As, M, K, a_sh, layout & 1)
    Bd, sb = stage(Bs, N, K, b_sh, layout & 2)
    sc = M * N + pad
    C = torch.full((batch * sc,), float("nan"), dtype=TORCH[out], device="cuda")
    g.gemm_plan_run_batched(plan, Ad.data_ptr(), Bd.data_ptr(), C.data_ptr(), batch, M, N, K, sa, sb, sc, dt, out,
                            layout, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert g.gemm_plan_status(plan) == 0
    C = C.cpu()
    if pad:
        assert bool(torch.isnan(C.view(batch, sc)[:, M * N:].float()).all()), "padding between outputs was written"
    return [C[e * sc:e * sc + M * N].view(M, N) for e in range(batch)]


def draw_batch(case, dist, dtype=wl.BF16, seed=0):
    batch, M, N, K, a_sh, b_sh, _, _ = case
    A, B = draw(M * (1 if a_sh else batch), N * (1 if b_sh else batch), K, dtype=dtype, dist=dist, seed=seed)
    As = A if a_sh else A.view(batch, M, K)
    Bs = B if b_sh else B.view(batch, N, K)
    return As, Bs


@pytest.mark.parametrize("unit", UNITS)
@pytest.mark.parametrize("case", BATCH_CASES, ids=lambda c: "b{}x{}x{}x{}".format(*c[:4]))
def test_batched_integer_bit_exact(g, plan, unit, case):
    batch, M, N, K, a_sh, b_sh, layout, pad = case
    configure(g, plan, unit)
    try:
        As, Bs = draw_batch(case, "int", seed=batch * 10 + unit)
        Cs = run_batched(g, plan, As, Bs, case, wl.F32)
        for e in range(batch):
            Ae = As if a_sh else As[e]
            Be = Bs if b_sh else Bs[e]
            C_ref, _ = oracle_full(Ae.contiguous(), Be.contiguous())
            assert np.array_equal(parity.to_f64(Cs[e]), C_ref), f"batch element {e}"
    finally:
        configure(g, plan, 4)


def test_batched_random_within_tolerance(g, plan):
    case = (3, 520, 776, 1008, False, False, 0, 0)   # K % 16 == 0 for the 8-bit case
    for dtype, out in ((wl.BF16, wl.BF16), (wl.F16, wl.F16), (wl.E4M3, wl.F32)):
        As, Bs = draw_batch(case, "normal", dtype=dtype, seed=7)
        Cs = run_batched(g, plan, As, Bs, case, out)
        for e in range(case[0]):
            C_ref, S = oracle_full(As[e].contiguous(), Bs[e].contiguous())
            parity.assert_within(parity.to_f64(Cs[e]), C_ref, S, out, f"batch {e} dtype {dtype}")


def test_bmm_helper_and_rules(g, plan):
    import ctypes
    A, B = draw(3 * 264, 200, 136, seed=5)
    A3 = A.view(3, 264, 136).cuda()
    C = g.bmm(A3, B.cuda(), plan, out_dtype=torch.float32)      # B shared
    torch.cuda.synchronize()
    for e in range(3):
        C_ref, S = oracle_full(A[e * 264:(e + 1) * 264], B)
        parity.assert_within(parity.to_f64(C[e]), C_ref, S, wl.F32, f"bmm {e}")
    vp = ctypes.c_void_p
    X = torch.zeros(4096, dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros(4096, dtype=torch.float32, device="cuda")
    args = (vp(plan), vp(X.data_ptr()), vp(X.data_ptr()), vp(Y.data_ptr()))
    rs = g.raw_status
    assert rs("gemm_plan_run_batched", *args, 2, 16, 16, 16, 256, 256, 200, 0, 2, 0, None) == g.GEMM_ERR_INVALID_ARG
    assert rs("gemm_plan_run_batched", *args, 2, 16, 16, 16, 260, 256, 256, 0, 2, 0, None) == g.GEMM_ERR_UNSUPPORTED
    assert rs("gemm_plan_run_batched", *args, -1, 16, 16, 16, 256, 256, 256, 0, 2, 0, None) == g.GEMM_ERR_INVALID_ARG
    assert rs("gemm_plan_run_batched", *args, 0, 16, 16, 16, 256, 256, 256, 0, 2, 0, None) == g.GEMM_OK
    torch.cuda.synchronize()
    assert g.gemm_plan_status(plan) == 0


# ------------------------------------------------------------------ full-size workloads

FULL = ["gemm_4096_bf16", "gemm_1024x4096x4096_f16", "gemm_ragged_4000x3000x5000", "gemm_8192_bf16",
        "gemm_4096_e4m3"]


def bench_launch(g, name):
    """The launch shape the benchmark times for workload `name` (its default
    plan), taken from gemm_plan_last_launch after one run on zero operands."""
    w = wl.WORKLOADS[name]
    h = g.gemm_plan_create(0)
    try:
        A = torch.zeros((w.M, w.K), dtype=TORCH[w.dtype], device="cuda")
        B = torch.zeros((w.N, w.K), dtype=TORCH[w.dtype], device="cuda")
        run(g, h, A, B, w.out_dtype)
        return g.gemm_plan_last_launch(h)
    finally:
        torch.cuda.synchronize()
        g.gemm_plan_destroy(h)


@pytest.mark.parametrize("name", FULL)
def test_workload_full_size(g, fresh_plan, name):
    """Full size, the benchmark's launch configuration (a default plan: same
    unit size, tile width, work list and grid as the timed launch, checked),
    every one of the M·N outputs against the fp64 oracle within the stated
    tolerance, element by element ("Chapter 7: Writing Custom Kernels with
    Pallas", §0/§2.3: each kernel checked against a float64 reference)."""
    w = wl.WORKLOADS[name]
    A, B = wl.make_inputs(w)
    C = run(g, fresh_plan, A.cuda(), B.cuda(), w.out_dtype)
    assert g.gemm_plan_last_launch(fresh_plan) == bench_launch(g, name)
    got = parity.to_f64(C)
    del C
    C_ref, S = oracle_full(A, B)
    parity.assert_within(got, C_ref, S, w.out_dtype, name)


@pytest.mark.parametrize("name,expect", [("gemm_4096_bf16", (2, 224, 152, 4)),
                                         ("gemm_8192_bf16", (2, 256, 224, 13))])
def test_default_launch_integer_bit_exact_full_size(g, fresh_plan, name, expect):
    """The default launches of the two square workloads -- 4096³: 76 CTA
    pairs, 256×224 tiles, 4 static waves; 8192³: 76 persistent pairs with 13
    waves of 256×256 tiles plus 36 one-tile clusters handed out at run time --
    on integer inputs in [-4, 4], with the workload's bf16 output.  Every
    partial sum is an integer below 16·K ≤ 2^17 < 2^24, exact in fp32, so each
    output must equal, bit for bit, the oracle's round-to-nearest-even of the
    exact sum."""
    w = wl.WORKLOADS[name]
    wi = wl.Workload(name + "_int", w.M, w.N, w.K, w.dtype, w.out_dtype, "int", w.seed, lo=-4, hi=4)
    A, B = wl.make_inputs(wi)
    C = run(g, fresh_plan, A.cuda(), B.cuda(), w.out_dtype)
    launch = g.gemm_plan_last_launch(fresh_plan)
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert (launch["ctas_per_unit"], launch["tile_n"], launch["ctas"], launch["dp_waves"]) == expect, launch
    got = parity.to_f64(C)
    del C
    C_ref, _ = oracle_full(A, B)
    want = oracle.decode(oracle.encode(C_ref, w.out_dtype), w.out_dtype)
    bad = got != want
    assert not bad.any(), f"{int(bad.sum())} of {bad.size} outputs differ; first at {tuple(np.argwhere(bad)[0])}"


def test_medium_ragged_full(g, plan):
    """The ragged workload's distribution and dtype, at a size the oracle
    finishes in seconds: several tiles in each direction, ragged in M, N and K."""
    w = wl.WORKLOADS["gemm_ragged_4000x3000x5000"]
    A, B = wl.make_inputs(w, M=1000, N=760, K=1256, seed=33)
    C = parity.to_f64(run(g, plan, A.cuda(), B.cuda(), w.out_dtype))
    C_ref, S = oracle_full(A, B)
    parity.assert_within(C, C_ref, S, w.out_dtype, "ragged 1000x760x1256")


def test_output_beyond_2_pow_32_elements(g, plan):
    """A C of more than 2^32 elements (66000 × 65600, bf16, 8.7 GB), ragged
    against every tile width, in the default launch: no 32-bit offset wraps
    anywhere between the host's tensor maps and the last tile's stores.
    Every element is written (C is NaN-poisoned and checked in row blocks);
    sampled entries, the corners and the tile edges match the oracle."""
    M, N, K = 66000, 65600, 64
    assert M * N > 1 << 32
    A, B = draw(M, N, K, seed=41)
    C = run(g, plan, A.cuda(), B.cuda(), wl.BF16)
    for r in range(0, M, 8192):
        assert bool(torch.isfinite(C[r:r + 8192]).all()), f"unwritten or non-finite entries in rows {r}.."
    I, J = parity.sample_positions(M, N, 2048, seed=41, tile_m=4096, tile_n=4096)
    got = C[torch.from_numpy(I).cuda(), torch.from_numpy(J).cuda()].to("cpu", torch.float64).numpy()
    del C
    C_ref, S = oracle.gemm_entries(wl.as_bits(A), wl.as_bits(B), wl.BF16, I, J)
    parity.assert_within(got, C_ref, S, wl.BF16, f"{M}x{N}x{K}")


# ------------------------------------------------------------------ edges and API behaviour

@pytest.mark.parametrize("unit", UNITS)
def test_long_k(g, plan, unit):
    """A K loop of 512 k-blocks (K = 32768) through a ring of 6-7 slots: the
    barrier phases wrap ~75 times.  Integer inputs keep every partial sum
    exact in fp32 (|sum| <= 16 K = 2^19), so the oracle's bits are the bar."""
    M, N, K = 256, 520, 32768
    configure(g, plan, unit)
    g.gemm_plan_set_option(plan, g.GEMM_OPT_SPLIT_K, 0)   # one K loop per tile, not slices
    try:
        A, B = draw(M, N, K, dist="int", seed=101)
        C = parity.to_f64(run(g, plan, A.cuda(), B.cuda(), wl.F32))
        C_ref, _ = oracle_full(A, B)
        assert np.array_equal(C, C_ref), f"{int((C != C_ref).sum())} mismatches"
    finally:
        configure(g, plan, 4)
        g.gemm_plan_set_option(plan, g.GEMM_OPT_SPLIT_K, -1)


def test_k_zero_writes_zeros(g, plan):
    for out in OUTS:
        A = torch.empty((37, 0), dtype=torch.bfloat16, device="cuda")
        B = torch.empty((48, 0), dtype=torch.bfloat16, device="cuda")
        C = run(g, plan, A, B, out)
        assert bool((C == 0).all())


def test_k_zero_batched_writes_zeros_only_in_the_products(g, plan):
    """K = 0 in a batch: every product is the empty sum, written in one
    launch; the gap between strided outputs stays untouched."""
    M, N, batch, sc = 37, 48, 3, 37 * 48 + 64
    A = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    C = torch.full((batch * sc,), float("nan"), dtype=torch.float32, device="cuda")
    g.gemm_plan_run_batched(plan, A.data_ptr(), A.data_ptr(), C.data_ptr(), batch, M, N, 0, 0, 0, sc, wl.BF16,
                            wl.F32, 0, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert g.gemm_plan_status(plan) == 0
    view = C.view(batch, sc)
    assert bool((view[:, :M * N] == 0).all())
    assert bool(torch.isnan(view[:, M * N:]).all())


def test_m_or_n_zero_is_noop(g, plan):
    A = torch.randn(0, 64, device="cuda").to(torch.bfloat16)
    B = torch.randn(16, 64, device="cuda").to(torch.bfloat16)
    C = torch.empty((0, 16), dtype=torch.float32, device="cuda")
    run(g, plan, A, B, wl.F32, C)
    A = torch.randn(16, 64, device="cuda").to(torch.bfloat16)
    sentinel = torch.full((4,), 7.0, device="cuda")
    g.gemm_plan_run(plan, A.data_ptr(), A.data_ptr(), sentinel.data_ptr(), 16, 0, 64, 0, 2, 0)
    torch.cuda.synchronize()
    assert bool((sentinel == 7.0).all())


@pytest.mark.parametrize("unit", UNITS)
def test_all_ones_ragged_is_k(g, fresh_plan, unit):
    """All-ones operands on a shape that is a multiple of no tile and of no
    k-block: every C[i,j] must be exactly K.  Out-of-bounds rows, columns and
    K elements of the last boxes arrive as zeros (TMA zero fill) and add
    nothing; any garbage there would show."""
    configure(g, fresh_plan, unit)
    for M, N, K, out in ((1000, 1096, 1000, wl.F32), (517, 264, 72, wl.BF16), (130, 1992, 4104, wl.F32)):
        A = torch.ones((M, K), dtype=torch.bfloat16, device="cuda")
        B = torch.ones((N, K), dtype=torch.bfloat16, device="cuda")
        C = run(g, fresh_plan, A, B, out).float()
        assert bool((C == K).all()), f"{M}x{N}x{K} unit={unit}: {int((C != K).sum())} entries differ from K"


def test_rows_beyond_m_untouched(g, plan):
    """C buffer has extra NaN rows past M: the clipped stores must not reach them."""
    M, N, K = 300, 264, 136
    A, B = draw(M, N, K, seed=5)
    for out in OUTS:
        buf = torch.full((M + 3, N), float("nan"), dtype=TORCH[out], device="cuda")
        run(g, plan, A.cuda(), B.cuda(), out, C=buf)
        assert bool(torch.isnan(buf[M:]).all())
        assert bool(torch.isfinite(buf[:M]).all())


def test_error_codes(g, plan):
    A = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((64, 64), dtype=torch.float32, device="cuda")
    rs = g.raw_status
    import ctypes
    vp = ctypes.c_void_p
    p = vp(plan)
    assert rs("gemm_plan_run", p, vp(A.data_ptr()), vp(A.data_ptr()), vp(C.data_ptr() + 4), 64, 64, 64, 0, 2,
              None) == g.GEMM_ERR_MISALIGNED
    assert rs("gemm_plan_run", p, vp(A.data_ptr()), vp(A.data_ptr()), vp(C.data_ptr()), 64, 64, 60, 0, 2,
              None) == g.GEMM_ERR_UNSUPPORTED
    assert rs("gemm_plan_run", p, vp(A.data_ptr()), vp(A.data_ptr()), vp(C.data_ptr()), 64, 6, 64, 0, 0,
              None) == g.GEMM_ERR_UNSUPPORTED
    assert rs("gemm_plan_run", p, vp(A.data_ptr()), vp(A.data_ptr()), vp(C.data_ptr()), 64, 64, 64, 2, 2,
              None) == g.GEMM_ERR_INVALID_ARG
    assert rs("gemm_plan_run", p, vp(A.data_ptr()), vp(A.data_ptr()), vp(C.data_ptr()), -1, 64, 64, 0, 2,
              None) == g.GEMM_ERR_INVALID_ARG
    assert rs("gemm_plan_set_option", p, 1, ctypes.c_int64(3)) == g.GEMM_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert g.gemm_plan_status(plan) == 0


def test_operands_must_be_device_memory_of_the_run_device(g, fresh_plan):
    """Host memory (pageable or pinned) where device memory belongs is refused
    by every run entry point before anything is encoded or launched:
    GEMM_ERR_INVALID_ARG, C untouched, the status word clear.  With K = 0 only
    C is read as an address.  Device operands then run as usual."""
    import ctypes
    vp = ctypes.c_void_p
    M, N, K = 256, 264, 128
    A, B = draw(M, N, K, dist="int", seed=7)
    Ad, Bd = A.cuda(), B.cuda()
    C = torch.full((M, N), float("nan"), device="cuda")
    Ch = torch.full((M, N), float("nan"))
    Ap, Chp = A.pin_memory(), Ch.pin_memory()
    pl, st = vp(fresh_plan), vp(torch.cuda.current_stream().cuda_stream)
    for a, b, c in ((A, Bd, C), (Ap, Bd, C), (Ad, B, C), (Ad, Bd, Ch), (Ad, Bd, Chp)):
        ptrs = (vp(a.data_ptr()), vp(b.data_ptr()), vp(c.data_ptr()))
        calls = {
            "gemm_plan_run": (pl, *ptrs, M, N, K, wl.BF16, wl.F32, st),
            "gemm_plan_run_layout": (pl, *ptrs, M, N, K, wl.BF16, wl.F32, 0, st),
            "gemm_plan_run_batched": (pl, *ptrs, 1, M, N, K, 0, 0, M * N, wl.BF16, wl.F32, 0, st),
            "gemm_run": (*ptrs, M, N, K, wl.BF16, wl.F32, st),
            "gemm_run_noalloc": (*ptrs, M, N, K, wl.BF16, wl.F32, st),
        }
        for fn, args in calls.items():
            assert g.raw_status(fn, *args) == g.GEMM_ERR_INVALID_ARG, (fn, a.device, b.device, c.device)
    # K = 0: C alone must be device memory
    assert g.raw_status("gemm_plan_run", pl, None, None, vp(Ch.data_ptr()), M, N, 0, wl.BF16, wl.F32, st) \
        == g.GEMM_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool(torch.isnan(C).all()) and bool(torch.isnan(Ch).all()) and bool(torch.isnan(Chp).all())
    assert g.gemm_plan_status(fresh_plan) == 0
    if torch.cuda.device_count() > 1:
        # a plan of device 1 refuses runs while device 0 is current
        other = g.gemm_plan_create(1)
        try:
            assert g.raw_status("gemm_plan_run", vp(other), vp(Ad.data_ptr()), vp(Bd.data_ptr()),
                                vp(C.data_ptr()), M, N, K, wl.BF16, wl.F32, st) == g.GEMM_ERR_INVALID_ARG
        finally:
            g.gemm_plan_destroy(other)
    got = parity.to_f64(run(g, fresh_plan, Ad, Bd, wl.F32, C))
    C_ref, _ = oracle_full(A, B)
    assert np.array_equal(got, C_ref)


def signed_permutation(n, seed):
    """An n×n matrix with one ±1 per row and column (a signed permutation)."""
    gen = torch.Generator().manual_seed(seed)
    perm = torch.randperm(n, generator=gen)
    sign = torch.randint(0, 2, (n,), generator=gen) * 2 - 1
    P = torch.zeros((n, n), dtype=torch.float32)
    P[torch.arange(n), perm] = sign.float()
    return P


# (M, K, options): one wave of 224-wide pair tiles; many waves with the
# partial last wave handed out at run time; the stream-K tail on a CTA cap;
# the 4-CTA multicast unit (K rows not a multiple of 128 bytes)
PDL_CHAINS = [(1024, 4096, {}), (4096, 2048, {9: 1}), (1300, 1096, {5: 1, 3: 14, 6: 0}), (1000, 1256, {6: 1})]


@pytest.mark.parametrize("pdl", [1, 0], ids=["pdl", "stream_order"])
@pytest.mark.parametrize("chain", PDL_CHAINS, ids=lambda c: f"{c[0]}x{c[1]}")
def test_back_to_back_chain_reads_each_result(g, fresh_plan, pdl, chain):
    """Sixteen products launched back to back on one stream, each reading the
    previous one's output as its A: X_{i+1} = X_i · P_iᵀ with P_i a signed
    permutation, so every X_i is a signed column permutation of X_0 (values
    in {-1, 0, 1}, exact in f16 at any length).  With programmatic dependent
    launch each grid may start while the previous one runs; it must still
    read the finished X_i.  Every intermediate is checked against the same
    permutations applied on the CPU."""
    M, K, opts = chain
    if opts.get(6) == 1 and torch.cuda.device_count() > 1:
        pytest.skip("the library multicasts only while one GPU is visible")
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_PDL, pdl)
    for k, v in opts.items():
        g.gemm_plan_set_option(fresh_plan, k, v)
    gen = torch.Generator().manual_seed(M + K)
    X0 = (torch.randint(0, 3, (M, K), generator=gen) - 1).to(torch.float16)
    Ps = [signed_permutation(K, 100 * M + i) for i in range(16)]
    xs = [X0.cuda()] + [torch.full((M, K), float("nan"), dtype=torch.float16, device="cuda") for _ in range(16)]
    Pd = [P.to(torch.float16).cuda() for P in Ps]
    st = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    for i in range(16):
        g.gemm_plan_run(fresh_plan, xs[i].data_ptr(), Pd[i].data_ptr(), xs[i + 1].data_ptr(), M, K, K, wl.F16,
                        wl.F16, st)
    torch.cuda.synchronize()
    assert g.gemm_plan_status(fresh_plan) == 0
    want = X0.float()
    for i in range(16):
        want = want @ Ps[i].t()
        got = xs[i + 1].float().cpu()
        assert torch.equal(got, want), f"product {i}: {int((got != want).sum())} entries differ"


def test_launch_right_after_torch_kernels_reads_their_output(g, fresh_plan):
    """Torch kernels rewrite A just before each launch (no programmatic
    signal from them): the product must see the rewritten A every time."""
    M, N, K = 1024, 1040, 1024
    A = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    B = torch.ones((N, K), dtype=torch.bfloat16, device="cuda")
    Cs = [torch.full((M, N), float("nan"), device="cuda") for _ in range(8)]
    st = torch.cuda.current_stream().cuda_stream
    for i in range(8):
        A.fill_(float(i - 3))                 # every entry i - 3: each C entry is K * (i - 3)
        g.gemm_plan_run(fresh_plan, A.data_ptr(), B.data_ptr(), Cs[i].data_ptr(), M, N, K, wl.BF16, wl.F32, st)
    torch.cuda.synchronize()
    assert g.gemm_plan_status(fresh_plan) == 0
    for i in range(8):
        assert bool((Cs[i] == K * (i - 3)).all()), i
    import ctypes
    for bad in (-1, 2):
        assert g.raw_status("gemm_plan_set_option", ctypes.c_void_p(fresh_plan), g.GEMM_OPT_PDL,
                            ctypes.c_int64(bad)) == g.GEMM_ERR_INVALID_ARG


# (M, N, K, input, output, split option): few tiles and a long K
SPLIT_CASES = [(256, 256, 8192, wl.BF16, wl.F32, -1), (128, 4096, 4096, wl.F16, wl.F16, -1),
               (384, 384, 4096, wl.BF16, wl.BF16, -1), (256, 512, 8192, wl.E4M3, wl.BF16, -1),
               (520, 264, 4096, wl.BF16, wl.F32, 8), (1000, 776, 2048, wl.F16, wl.F32, 2)]


@pytest.mark.parametrize("case", SPLIT_CASES, ids=lambda c: "x".join(map(str, c[:3])) + f"_s{c[5]}")
def test_split_k_products(g, fresh_plan, case):
    """Products with few tiles and a long K run as K slices (fp32 partials in
    the workspace) plus an in-order reduction: split chosen automatically or
    forced, the result on integer inputs equal bit for bit to the unsplit
    product and to the oracle, on random inputs within the tolerance, and
    the same bits twice."""
    M, N, K, dt, out, split = case
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_SPLIT_K, split)
    A, B = draw(M, N, K, dtype=dt, dist="int", seed=M + K)
    Ad, Bd = A.cuda(), B.cuda()
    C = run(g, fresh_plan, Ad, Bd, out)
    assert g.gemm_plan_last_split(fresh_plan) > 1, "not split"
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_SPLIT_K, 0)
    C1 = run(g, fresh_plan, Ad, Bd, out)
    assert g.gemm_plan_last_split(fresh_plan) == 1
    assert torch.equal(C, C1), "split and unsplit products differ on integer inputs"
    C_ref, _ = oracle_full(A, B)
    want = C_ref if out == wl.F32 else oracle.decode(oracle.encode(C_ref, out), out)
    assert np.array_equal(parity.to_f64(C), want)
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_SPLIT_K, split)
    A, B = draw(M, N, K, dtype=dt, seed=M + K + 1)
    Ad, Bd = A.cuda(), B.cuda()
    C = run(g, fresh_plan, Ad, Bd, out)
    C2 = run(g, fresh_plan, Ad, Bd, out)
    assert torch.equal(C, C2), "split product not repeatable"
    C_ref, S = oracle_full(A, B)
    parity.assert_within(parity.to_f64(C), C_ref, S, out, f"split {case}")


def test_split_k_rules(g, fresh_plan):
    """No split where it cannot pay or is not allowed: many tiles, short K,
    K not a whole number of k-blocks, MN-major operands, option 0."""
    import ctypes
    for M, N, K in ((4096, 4096, 4096), (256, 256, 256), (256, 256, 8200)):
        A = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
        B = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
        run(g, fresh_plan, A, B, wl.F32)
        assert g.gemm_plan_last_split(fresh_plan) == 1, (M, N, K)
    A, B = draw(256, 256, 8192, seed=5)
    C = run_layout(g, fresh_plan, A.cuda(), B.cuda(), 2, wl.F32)
    assert g.gemm_plan_last_split(fresh_plan) == 1
    C_ref, S = oracle_full(A, B)
    parity.assert_within(parity.to_f64(C), C_ref, S, wl.F32, "MN-major B, not split")
    for bad in (1, 3, 64, -2):
        assert g.raw_status("gemm_plan_set_option", ctypes.c_void_p(fresh_plan), g.GEMM_OPT_SPLIT_K,
                            ctypes.c_int64(bad)) == g.GEMM_ERR_INVALID_ARG


def test_split_k_from_two_streams_on_one_plan(g, fresh_plan):
    """Split products share the plan's workspace: issued from two streams at
    once they are ordered on the GPU by the library, so every result is
    exact."""
    M, N, K = 256, 256, 8192
    data = [draw(M, N, K, dist="int", seed=300 + i) for i in range(2)]
    refs = [oracle_full(A, B)[0] for A, B in data]
    dev = [(A.cuda(), B.cuda()) for A, B in data]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [[], []]
    for _ in range(20):
        for i in range(2):
            C = torch.full((M, N), float("nan"), device="cuda")
            g.gemm_plan_run(fresh_plan, dev[i][0].data_ptr(), dev[i][1].data_ptr(), C.data_ptr(), M, N, K, wl.BF16,
                            wl.F32, streams[i].cuda_stream)
            outs[i].append(C)
    torch.cuda.synchronize()
    assert g.gemm_plan_status(fresh_plan) == 0
    assert g.gemm_plan_last_split(fresh_plan) > 1
    for i in range(2):
        for C in outs[i]:
            assert np.array_equal(parity.to_f64(C), refs[i]), f"stream {i}"


def test_split_k_in_cuda_graph(g, fresh_plan):
    """A split product (slices and reduction) recorded into a CUDA graph and
    replayed on new integer inputs equals the oracle every time."""
    M, N, K = 384, 384, 4096
    Ad = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    Bd = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    Cd = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g.gemm_plan_run(fresh_plan, Ad.data_ptr(), Bd.data_ptr(), Cd.data_ptr(), M, N, K, wl.BF16, wl.F32,
                        s.cuda_stream)
    s.synchronize()
    assert g.gemm_plan_last_split(fresh_plan) > 1
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        g.gemm_plan_run(fresh_plan, Ad.data_ptr(), Bd.data_ptr(), Cd.data_ptr(), M, N, K, wl.BF16, wl.F32,
                        s.cuda_stream)
    for rep in range(3):
        A, B = draw(M, N, K, dist="int", seed=70 + rep)
        Ad.copy_(A)
        Bd.copy_(B)
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(parity.to_f64(Cd), oracle_full(A, B)[0]), rep
    assert g.gemm_plan_status(fresh_plan) == 0


def test_clock_log_records_each_launch(g, fresh_plan):
    """GEMM_OPT_CLOCK_LOG keeps, per launch, the SM cycles and nanoseconds of
    the first CTA's lifetime: one record per launch, oldest first, a
    plausible SM clock, the most recent `value` launches when more ran, and
    the log empty once read."""
    import ctypes
    M, N, K = 2048, 2048, 4096
    A, B = draw(M, N, K, seed=17)
    Ad, Bd = A.cuda(), B.cuda()
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    vp = ctypes.c_void_p
    n = ctypes.c_int64(0)
    assert g.raw_status("gemm_plan_clock_log", vp(fresh_plan), None, 0, ctypes.byref(n)) == g.GEMM_ERR_UNSUPPORTED
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_CLOCK_LOG, 8)
    for _ in range(5):
        run(g, fresh_plan, Ad, Bd, wl.BF16, C)
    recs = g.gemm_plan_clock_log(fresh_plan)
    assert len(recs) == 5, recs
    props = torch.cuda.get_device_properties(0)
    for cycles, ns in recs:
        assert ns > 1000 and cycles > 0, recs
        assert 200.0 < cycles / ns * 1e3 < 3000.0, recs   # MHz
    assert g.gemm_plan_clock_log(fresh_plan) == []
    for _ in range(11):
        run(g, fresh_plan, Ad, Bd, wl.BF16, C)
    assert len(g.gemm_plan_clock_log(fresh_plan)) == 8
    assert len(g.gemm_plan_clock_log(fresh_plan, capacity=3)) == 0
    run(g, fresh_plan, Ad, Bd, wl.BF16, C)
    run(g, fresh_plan, Ad, Bd, wl.BF16, C)
    assert len(g.gemm_plan_clock_log(fresh_plan, capacity=1)) == 1
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_CLOCK_LOG, 0)
    run(g, fresh_plan, Ad, Bd, wl.BF16, C)
    assert g.raw_status("gemm_plan_clock_log", vp(fresh_plan), None, 0, ctypes.byref(n)) == g.GEMM_ERR_UNSUPPORTED
    for bad in (-1, (1 << 20) + 1):
        assert g.raw_status("gemm_plan_set_option", vp(fresh_plan), g.GEMM_OPT_CLOCK_LOG, ctypes.c_int64(bad)) \
            == g.GEMM_ERR_INVALID_ARG
    del props


DEBUG_RUN = r"""
import sys, numpy as np, torch
sys.path.insert(0, {root!r})
import dense_gemm_blackwell_persistent_gb300 as g
import oracle, workloads as wl
assert g.VARIANT == "debug" and g.LIB_PATH.endswith("_debug.so"), g.LIB_PATH
torch.cuda.set_device(0)
# (M, N, K, in, out, options, layout, batch)
cases = [
    (1000, 776, 1256, wl.BF16, wl.F32, {{}}, 0, 1),                                # 4-CTA multicast unit
    (1024, 1040, 1024, wl.F16, wl.BF16, {{}}, 0, 1),                              # CTA pairs
    (520, 776, 392, wl.BF16, wl.F32, {{g.GEMM_OPT_CTA_PAIR: 1}}, 0, 1),           # single CTAs
    (1300, 1096, 520, wl.BF16, wl.F32, {{g.GEMM_OPT_DYNAMIC: 2}}, 0, 1),          # every tile handed out
    (1300, 1096, 2000, wl.BF16, wl.F32, {{g.GEMM_OPT_STREAM_K: 1, g.GEMM_OPT_MAX_CTAS: 14,
                                          g.GEMM_OPT_MULTICAST: 0}}, 0, 1),                # stream-K tail
    (264, 200, 136, wl.BF16, wl.F16, {{}}, 0, 3),                                 # batched
    (384, 448, 264, wl.BF16, wl.F32, {{}}, 3, 1),                                 # A K×M, B K×N
    (512, 384, 1024, wl.E4M3, wl.BF16, {{}}, 0, 1),                               # 8-bit operands
]
for M, N, K, dt, out, opts, layout, batch in cases:
    plan = g.gemm_plan_create(0)
    for k, v in opts.items():
        g.gemm_plan_set_option(plan, k, v)
    w = wl.Workload("dbg", M * batch, N, K, dt, out, "int", M + N + K, lo=-4, hi=4)
    A, Bfull = wl.make_inputs(w, N=N * batch)
    As = A.view(batch, M, K)
    Bs = Bfull.view(batch, N, K)
    Ad = (As.transpose(1, 2) if layout & 1 else As).contiguous().cuda()
    Bd = (Bs.transpose(1, 2) if layout & 2 else Bs).contiguous().cuda()
    C = torch.full((batch, M, N), float("nan"), dtype=wl.TORCH_DTYPES[out], device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    g.gemm_plan_run_batched(plan, Ad.data_ptr(), Bd.data_ptr(), C.data_ptr(), batch, M, N, K, M * K, N * K, M * N,
                            dt, out, layout, s)
    torch.cuda.synchronize()
    st = g.gemm_plan_status(plan)
    assert st == 0, (M, N, K, opts, st, g.gemm_strerror(st))
    for e in range(batch):
        ref, _ = oracle.gemm(wl.as_bits(As[e]), wl.as_bits(Bs[e]), dt)
        want = ref if out == wl.F32 else oracle.decode(oracle.encode(ref, out), out)
        got = C[e].to("cpu", torch.float64).numpy()
        assert np.array_equal(got, want), (M, N, K, opts, e)
    g.gemm_plan_destroy(plan)
print("debug build: every case status 0 and exact")
"""


def test_debug_build_normal_runs_report_status_zero():
    """The GEMM_DEBUG variant checks, inside the kernel, every work item's tile
    and k-block range, the tile coordinates and operand rows of each load,
    the ring's stage and phase, the accumulator buffer and every store box,
    recording GEMM_ERR_INTERNAL instead of making the access.  On correct
    runs -- every unit size, the dynamic list, stream-K, a batch, MN-major
    operands, 8-bit operands -- it must record nothing, and the results are
    exact on integer inputs.  Runs in a child process that loads that
    variant."""
    import os
    import subprocess
    import sys
    from dense_gemm_blackwell_persistent_gb300 import _build
    _build.build(variant="debug")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, GB300_GEMM_VARIANT="debug")
    res = subprocess.run([sys.executable, "-c", DEBUG_RUN.format(root=root)], env=env, capture_output=True,
                         text=True, timeout=600)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-4000:]
    assert "every case status 0 and exact" in res.stdout


@pytest.mark.parametrize("dynamic", [0, 2], ids=["static", "dynamic"])
@pytest.mark.parametrize("unit", UNITS)
def test_bounded_wait_expires_and_plan_recovers(g, fresh_plan, unit, dynamic):
    """Failure detection without a GPU fault: with the test option on, the MMA
    warp waits on a barrier nothing completes.  The wait runs out after the
    shortened bound, the kernel records GEMM_ERR_TIMEOUT, the other roles
    leave their loops (abort flag, or their own bound in the peer CTAs), the
    CTAs tear down in order, and the same plan then computes correctly."""
    import time
    configure(g, fresh_plan, unit)
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_DYNAMIC, dynamic)
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_WAIT_LIMIT_US, 20000)   # 20 ms
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_STALL_TEST, 1)
    A, B = draw(512, 520, 512, dist="int", seed=9)
    Ad, Bd = A.cuda(), B.cuda()
    C = torch.full((512, 520), float("nan"), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    g.gemm_plan_run(fresh_plan, Ad.data_ptr(), Bd.data_ptr(), C.data_ptr(), 512, 520, 512, wl.BF16, wl.F32,
                    torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert g.gemm_plan_status(fresh_plan) == g.GEMM_ERR_TIMEOUT
    assert elapsed < 2.0, f"the timeout path took {elapsed:.2f} s for a 20 ms bound"
    assert g.gemm_plan_status(fresh_plan) == g.GEMM_OK, "status is cleared once read"
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_STALL_TEST, 0)
    C = parity.to_f64(run(g, fresh_plan, Ad, Bd, wl.F32))
    C_ref, _ = oracle_full(A, B)
    assert np.array_equal(C, C_ref)


def test_encoder_failure_is_reported_before_any_launch(g, fresh_plan):
    """Failure detection on the host: with the test option on, the driver's
    tensor-map encoder is replaced by a fake that rejects the map.  The run
    must return GEMM_ERR_DRIVER, launch nothing (C keeps its NaN poison, the
    last launch record is unchanged, the device status is clean), and the
    same plan must compute correctly once the option is off."""
    M, N, K = 300, 264, 136
    A, B = draw(M, N, K, dist="int", seed=61)
    Ad, Bd = A.cuda(), B.cuda()
    run(g, fresh_plan, Ad, Bd, wl.F32)
    before = g.gemm_plan_last_launch(fresh_plan)
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_FAIL_ENCODE, 1)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    with pytest.raises(g.GemmError) as e:
        g.gemm_plan_run(fresh_plan, Ad.data_ptr(), Bd.data_ptr(), C.data_ptr(), M, N, K, wl.BF16, wl.F32,
                        torch.cuda.current_stream().cuda_stream)
    assert e.value.status == g.GEMM_ERR_DRIVER
    torch.cuda.synchronize()
    assert bool(torch.isnan(C).all()), "a rejected run wrote C"
    assert g.gemm_plan_last_launch(fresh_plan) == before
    assert g.gemm_plan_status(fresh_plan) == g.GEMM_OK
    g.gemm_plan_set_option(fresh_plan, g.GEMM_OPT_FAIL_ENCODE, 0)
    C_ref, _ = oracle_full(A, B)
    assert np.array_equal(parity.to_f64(run(g, fresh_plan, Ad, Bd, wl.F32)), C_ref)


def test_wait_options_are_checked(g, fresh_plan):
    import ctypes
    p = ctypes.c_void_p(fresh_plan)
    assert g.raw_status("gemm_plan_set_option", p, g.GEMM_OPT_WAIT_LIMIT_US, ctypes.c_int64(-1)) \
        == g.GEMM_ERR_INVALID_ARG
    assert g.raw_status("gemm_plan_set_option", p, g.GEMM_OPT_WAIT_LIMIT_US, ctypes.c_int64(60000001)) \
        == g.GEMM_ERR_INVALID_ARG
    assert g.raw_status("gemm_plan_set_option", p, g.GEMM_OPT_STALL_TEST, ctypes.c_int64(2)) \
        == g.GEMM_ERR_INVALID_ARG


def test_implicit_plan_and_host_entry_agree(g, plan):
    M, N, K = 520, 776, 392
    A, B = draw(M, N, K, dtype=wl.F16, seed=9)
    C1 = run(g, plan, A.cuda(), B.cuda(), wl.BF16)
    # gemm_run uses the plan most recently created on the device
    C2 = torch.full_like(C1, float("nan"))
    Ad, Bd = A.cuda(), B.cuda()
    g.gemm_run(Ad.data_ptr(), Bd.data_ptr(), C2.data_ptr(), M, N, K, wl.F16, wl.BF16,
               torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))
    # host buffers in, host buffer out
    Ah, Bh = A.pin_memory(), B.pin_memory()
    C3 = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    g.gemm_plan_run_host(plan, Ah.data_ptr(), Bh.data_ptr(), C3.data_ptr(), M, N, K, wl.F16, wl.BF16,
                         torch.cuda.current_stream().cuda_stream)
    assert torch.equal(C1.cpu().view(torch.int16), C3.view(torch.int16))


@pytest.mark.parametrize("shape", [(2100, 520, 264), (1024, 776, 392), (4096, 264, 136)])
def test_host_entry_pipelined_chunks(g, fresh_plan, shape):
    """gemm_plan_run_host splits A into row chunks (copies, products and
    copies back overlapped on the plan's streams): integer inputs give the
    oracle's bits for every chunk, including a ragged last one, and the
    caller's stream sees the finished C."""
    M, N, K = shape
    A, B = draw(M, N, K, dist="int", seed=M + N)
    Ah, Bh = A.pin_memory(), B.pin_memory()
    for out in (wl.F32, wl.BF16):
        Ch = torch.full((M, N), float("nan"), dtype=TORCH[out]).pin_memory()
        g.gemm_plan_run_host(fresh_plan, Ah.data_ptr(), Bh.data_ptr(), Ch.data_ptr(), M, N, K, wl.BF16, out,
                             torch.cuda.current_stream().cuda_stream)
        assert g.gemm_plan_status(fresh_plan) == 0
        C_ref, _ = oracle_full(A, B)
        want = C_ref if out == wl.F32 else oracle.decode(oracle.encode(C_ref, out), out)
        assert np.array_equal(parity.to_f64(Ch), want), f"{shape} out={out}"


def test_deterministic(g, plan):
    w = wl.WORKLOADS["gemm_1024x4096x4096_f16"]
    A, B = wl.make_inputs(w)
    Ad, Bd = A.cuda(), B.cuda()
    C1 = run(g, plan, Ad, Bd, w.out_dtype)
    C2 = run(g, plan, Ad, Bd, w.out_dtype)
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))


def test_helpers_without_a_plan(g):
    """matmul() and bmm() without a plan use one default plan per device,
    created on first use and reused."""
    A, B = draw(264, 200, 136, dist="int", seed=71)
    C = g.matmul(A.cuda(), B.cuda(), out_dtype=torch.float32)
    torch.cuda.synchronize()
    C_ref, _ = oracle_full(A, B)
    assert np.array_equal(parity.to_f64(C), C_ref)
    assert g.default_plan() == g.default_plan(0) == g.default_plan(torch.device("cuda", 0))
    C3 = g.bmm(A.cuda().view(1, 264, 136), B.cuda(), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert np.array_equal(parity.to_f64(C3[0]), C_ref)


def test_torch_matmul_helper(g, plan):
    A, B = draw(256, 512, 128, seed=3)
    Ad, Bd = A.cuda(), B.cuda()
    C = g.matmul(Ad, Bd, out_dtype=torch.float32, plan=plan)
    torch.cuda.synchronize()
    C_ref, S = oracle_full(A, B)
    parity.assert_within(parity.to_f64(C), C_ref, S, wl.F32, "matmul helper")


def test_plain_c_caller_bit_exact(g, tmp_path):
    """A C99 program with no CUDA headers (tests/native/c_caller.c) runs a
    ragged integer product through gemm_plan_run_host and checks every
    element against an exact integer loop, then checks that bad arguments
    come back as codes."""
    import subprocess
    from tests.test_abi import build_c_caller
    exe = str(tmp_path / "c_caller")
    build_c_caller(g.LIB_PATH, exe)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c caller ok" in r.stdout
