"""The kernel's work schedule (csrc/schedule.h), checked on the CPU.

The same header the kernel compiles is built here with g++ into a small
driver that prints every unit's work items.  For many (tiles, units,
k-blocks) combinations, including the benchmark shapes on 76 CTA pairs, the
tests check that every (tile, k-block) is computed exactly once, that the
data-parallel part is balanced and the stream-K tail splits its k-blocks
evenly, and that the split-tile bookkeeping the epilogue relies on
(contributor order, contributor count, workspace slots, counters) is
consistent.
"""
import os
import subprocess
from collections import defaultdict

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "dense_gemm_blackwell_persistent_gb300", "csrc")
SRC = os.path.join(ROOT, "tests", "native", "schedule_dump.cpp")


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
                cur = {"sched": tuple(map(int, f[1:])), "work": [], "contrib_slots": {}}
            elif f[0] == "W":
                cur["work"].append(tuple(map(int, f[1:])))
            elif f[0] == "C":
                q, c, slot = map(int, f[1:])
                cur["contrib_slots"][(q, c)] = slot
            elif f[0] == "E":
                results.append(cur)
        return results
    return run


def check(res, tiles, units, kb, allow):
    T, P, KB, W, R = res["sched"]
    assert (T, P, KB) == (tiles, units, kb)
    cover = defaultdict(int)
    per_unit_kblocks = defaultdict(int)
    tile_contribs = defaultdict(list)
    slots_used = set()
    for (u, j, tile, kb0, kb1, c, n, slot, q) in res["work"]:
        assert 0 <= u < P and 0 <= tile < T and 0 <= kb0 < kb1 <= KB
        for k in range(kb0, kb1):
            cover[(tile, k)] += 1
        per_unit_kblocks[u] += kb1 - kb0
        if n == 1:
            assert (kb0, kb1) == (0, KB), "an unsplit tile must cover all of K"
        else:
            assert R > 0 and tile >= W * P and q == tile - W * P
            assert slot in (2 * u, 2 * u + 1)
            assert slot not in slots_used, "a workspace slot is reused within a launch"
            slots_used.add(slot)
            tile_contribs[tile].append((c, n, kb0, u, slot))
    # every (tile, k-block) exactly once
    assert len(cover) == T * KB and set(cover.values()) == {1}
    # split tiles: contributors 0..n-1 in k order, slots found by contributor_slot
    for tile, lst in tile_contribs.items():
        lst.sort()
        n = lst[0][1]
        assert [c for c, *_ in lst] == list(range(n)) and all(x[1] == n for x in lst)
        assert [kb0 for _, _, kb0, _, _ in lst] == sorted(kb0 for _, _, kb0, _, _ in lst)
        q = tile - W * P
        for c, _, _, u, slot in lst:
            assert res["contrib_slots"][(q, c)] == slot
    if R == 0:
        assert W == -(-T // P)
        loads = [per_unit_kblocks[u] for u in range(P)]
        assert max(loads) - min(loads) <= KB
    else:
        assert allow and W == T // P and R == T - W * P and R * 8 <= P * 7
        tail = [per_unit_kblocks[u] - W * KB for u in range(P)]
        assert max(tail) - min(tail) <= 1 and min(tail) >= 2, tail


BENCH_CASES = [
    (256, 76, 64, True),     # bf16 4096^3, 256x256 tiles on 76 pairs
    (64, 76, 64, True),      # f16 1024x4096x4096: fewer tiles than pairs
    (192, 76, 79, True),     # ragged 4000x3000x5000 (K tail block)
    (1024, 76, 128, True),   # bf16 8192^3
    (1, 76, 4, True),        # 256^3
    (256, 76, 64, False),
    (1024, 76, 128, False),
]


def test_benchmark_shapes(dump):
    for case, res in zip(BENCH_CASES, dump(BENCH_CASES)):
        check(res, *case)


def test_expected_splits(dump):
    res = dump([(256, 76, 64, True), (64, 76, 64, True), (1, 76, 4, True), (76, 76, 64, True)])
    assert res[0]["sched"][3:] == (3, 28)    # 3 full waves + 28 tiles spread over all pairs
    assert res[1]["sched"][3:] == (0, 64)    # all 64 tiles spread over 76 pairs
    assert res[2]["sched"][3:] == (1, 0)     # too little work to split
    assert res[3]["sched"][3:] == (1, 0)     # exactly one full wave


def test_random_shapes(dump):
    rng = np.random.default_rng(0)
    cases = []
    for _ in range(400):
        P = int(rng.integers(1, 160))
        T = int(rng.integers(1, 6 * P + 3))
        KB = int(rng.integers(1, 200))
        cases.append((T, P, KB, bool(rng.integers(0, 4) > 0)))
    for case, res in zip(cases, dump(cases)):
        check(res, *case)
