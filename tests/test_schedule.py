"""The kernel's work schedule (csrc/schedule.h), checked on the CPU.

The same header the kernel compiles is built here with g++ into a small
driver that prints every unit's work items.  For many (tiles, units,
k-blocks) combinations, including the benchmark shapes on 76 CTA pairs, the
tests check that every (tile, k-block) is computed exactly once, that the
whole-tile waves are balanced and the stream-K part splits its k-blocks
evenly, and the invariants the epilogue's fix-up relies on: a tile has at
most two pieces; the piece with the tile's first k-blocks is its unit's last
work item and finishes the tile; the other is its unit's first stream-K
item; both name the same workspace slot (the second piece's unit) and the
same flag; no slot or flag is used twice in a launch.  For the dynamic work
list (cluster launch control) they check that the clusters' lists cover
every tile exactly once.
"""
import os
import subprocess
from collections import defaultdict

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "dense_gemm_blackwell_persistent_gb300", "csrc")
SRC = os.path.join(ROOT, "tests", "native", "schedule_dump.cpp")
FIXUP_KBLOCKS = 12  # kFixupKBlocks in schedule.h


@pytest.fixture(scope="module")
def dump(tmp_path_factory):
    exe = str(tmp_path_factory.mktemp("sched") / "schedule_dump")
    subprocess.run(["g++", "-O1", "-std=c++17", "-I", CSRC, SRC, "-o", exe], check=True)

    def run(cases):
        inp = "".join(f"{t} {u} {k} {int(a)}\n" for t, u, k, a in cases)
        out = subprocess.run([exe], input=inp, capture_output=True, text=True, check=True).stdout
        results, cur = [], None
        for line in out.splitlines():
            f = line.split()
            if f[0] == "S":
                cur = {"sched": tuple(map(int, f[1:])), "work": []}
            elif f[0] == "W":
                cur["work"].append(tuple(map(int, f[1:])))
            elif f[0] == "E":
                results.append(cur)
        return results
    return run


def expected_mode(T, P, KB, allow):
    """Which schedule the rule in schedule.h picks: 'dp', 'wave' or 'halves'."""
    W, R = divmod(T, P)
    if allow and R and KB >= 2:
        if W >= 1 and (P - R) * KB > FIXUP_KBLOCKS * P:
            return "wave"
        if W == 0 and 2 * T <= P and KB > 2 * FIXUP_KBLOCKS:
            return "halves"
    return "dp"


def check(res, tiles, units, kb, allow):
    T, P, KB, W, S = res["sched"]
    assert (T, KB) == (tiles, kb)
    mode = expected_mode(tiles, units, kb, allow)
    if mode == "dp":
        assert S == 0 and P == max(1, min(units, tiles)) and W == -(-T // P)
    elif mode == "wave":
        assert P == units and W == tiles // units - 1 and S == units + tiles % units
    else:
        assert P == 2 * tiles and W == 0 and S == tiles
    cover = defaultdict(int)
    per_unit_sk = defaultdict(int)
    items = defaultdict(list)
    pieces = defaultdict(list)
    for (u, j, tile, kb0, kb1, c, n, slot, q) in res["work"]:
        assert 0 <= u < P and 0 <= tile < T and 0 <= kb0 < kb1 <= KB
        items[u].append(j)
        for k in range(kb0, kb1):
            cover[(tile, k)] += 1
        if j >= W and S:
            per_unit_sk[u] += kb1 - kb0
            assert tile == W * P + q
        if n == 1:
            assert (kb0, kb1) == (0, KB) and slot == -1, "an unsplit tile must cover all of K"
        else:
            assert n == 2 and S > 0 and c in (0, 1)
            pieces[tile].append((c, u, j, kb0, kb1, slot, q))
    # every (tile, k-block) exactly once
    assert len(cover) == T * KB and set(cover.values()) == {1}
    last_item = {u: max(js) for u, js in items.items()}
    slots, flags = set(), set()
    for tile, lst in pieces.items():
        lst.sort()
        assert [c for c, *_ in lst] == [0, 1], lst
        (_, u0, j0, a0, b0, s0, q0), (_, u1, j1, a1, b1, s1, q1) = lst
        assert a0 == 0 and b0 == a1 and b1 == KB, "the two pieces split K at one point"
        assert j0 == last_item[u0], "the finishing piece is its unit's last item"
        assert j1 == W, "the other piece is its unit's first stream-K item"
        assert s0 == s1 == u1 and q0 == q1
        assert s1 not in slots and q1 not in flags
        slots.add(s1)
        flags.add(q1)
        assert 0 <= q1 < 2 * P
    if S:
        loads = [per_unit_sk[u] for u in range(P)]
        assert max(loads) - min(loads) <= 1, loads
        if mode == "wave":
            assert min(loads) >= KB, "every stream-K range is longer than a tile"
    else:
        loads = [len(items[u]) for u in range(P)]
        assert max(loads) - min(loads) <= 1


BENCH_CASES = [
    (304, 76, 64, True),     # bf16 4096^3, 256x224 tiles on 76 pairs: 4 whole waves
    (256, 76, 64, True),     # bf16 4096^3, 256x256 tiles: 3.4 waves
    (76, 76, 64, True),      # f16 1024x4096x4096, 256x224 tiles: one whole wave
    (96, 36, 79, True),      # ragged 4000x3000x5000 on 36 four-CTA clusters (K tail block)
    (1024, 76, 128, True),   # bf16 8192^3
    (1, 76, 4, True),        # 256^3
    (256, 76, 64, False),
    (1024, 76, 128, False),
]


def test_benchmark_shapes(dump):
    for case, res in zip(BENCH_CASES, dump(BENCH_CASES)):
        check(res, *case)


def test_expected_splits(dump):
    res = dump([(256, 76, 64, True), (1024, 76, 128, True), (20, 76, 32, True), (1, 76, 4, True),
                (76, 76, 64, True), (150, 76, 64, True), (40, 76, 64, True), (144, 76, 48, True)])
    assert res[0]["sched"][1:] == (76, 64, 2, 104)   # 2 whole waves + 76 + 28 tiles spread over all pairs
    assert res[1]["sched"][1:] == (76, 128, 12, 112)  # 8192^3: 12 whole waves + 112 tiles spread
    assert res[2]["sched"][1:] == (40, 32, 0, 20)    # 20 tiles halved over 40 units
    assert res[3]["sched"][1:] == (1, 4, 1, 0)       # too little K to split
    assert res[4]["sched"][1:] == (76, 64, 1, 0)     # exactly one whole wave
    assert res[5]["sched"][1:] == (76, 64, 2, 0)     # 74 of 76 in the last wave: splitting would not pay
    assert res[6]["sched"][1:] == (40, 64, 1, 0)     # more than half the units: whole tiles
    assert res[7]["sched"][1:] == (76, 48, 2, 0)     # 3072^3: 68 of 76 in the last wave, short K


def test_random_shapes(dump):
    rng = np.random.default_rng(0)
    cases = []
    for _ in range(600):
        P = int(rng.integers(1, 160))
        T = int(rng.integers(1, 6 * P + 3))
        KB = int(rng.integers(1, 200))
        cases.append((T, P, KB, bool(rng.integers(0, 4) > 0)))
    for case, res in zip(cases, dump(cases)):
        check(res, *case)


@pytest.fixture(scope="module")
def dump_raw(tmp_path_factory):
    exe = str(tmp_path_factory.mktemp("sched_dyn") / "schedule_dump")
    subprocess.run(["g++", "-O1", "-std=c++17", "-I", CSRC, SRC, "-o", exe], check=True)

    def run(cases):
        inp = "".join(f"{t} {u} {w} -1\n" for t, u, w in cases)
        out = subprocess.run([exe], input=inp, capture_output=True, text=True, check=True).stdout
        results, cur = [], None
        for line in out.splitlines():
            f = line.split()
            if f[0] == "D":
                cur = {"head": tuple(map(int, f[1:])), "lists": defaultdict(list)}
            elif f[0] == "L":
                c, k, tile = map(int, f[1:])
                assert k == len(cur["lists"][c])
                cur["lists"][c].append(tile)
            elif f[0] == "E":
                results.append(cur)
        return results
    return run


def dynamic_cases():
    """(tiles, units, waves) as the host builds them: the partial last wave
    handed out (units = resident units, waves = tiles // units, tiles not a
    multiple), and every tile a list (units = tiles, waves = 1)."""
    cases = []
    for T in (77, 112, 304 + 5, 1024, 1184, 512, 6, 1):
        for P in (76, 36, 152, 5):
            if T > P and T % P:
                cases.append((T, P, T // P))
        cases.append((T, T, 1))
    return cases


def test_dynamic_lists_cover_every_tile_once(dump_raw):
    """Every tile belongs to exactly one cluster's list, the persistent
    clusters own the static raster's whole waves (c, c + P, ...), and each
    tile of the partial wave is a list of its own."""
    cases = dynamic_cases()
    for (T, P, D), res in zip(cases, dump_raw(cases)):
        t, u, w, n = res["head"]
        assert (t, u, w) == (T, P, D) and n == P + (T - P * D)
        owner = {}
        for c in range(n):
            lst = res["lists"][c]
            if c < P:
                assert lst == [c + k * P for k in range(D)], (T, P, D, c)
            else:
                assert lst == [P * D + (c - P)], (T, P, D, c)
            for tile in lst:
                assert tile not in owner, (T, P, D, tile)
                owner[tile] = c
        assert sorted(owner) == list(range(T)), (T, P, D)


def test_fast_division_matches_the_operator(tmp_path):
    """The multiply-and-shift divider the kernel decodes tiles with equals
    integer division for every divisor up to 5000 and for divisors near
    every power of two and at random up to 2^31 - 1, on numerators at the
    edges of the range and at random."""
    exe = str(tmp_path / "fastdiv_check")
    subprocess.run(["g++", "-O1", "-std=c++17", "-I", CSRC, os.path.join(ROOT, "tests", "native", "fastdiv_check.cpp"),
                    "-o", exe], check=True)
    out = subprocess.run([exe], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.startswith("ok "), out.stdout + out.stderr
    assert int(out.stdout.split()[1]) > 1_000_000
