"""The launch shape the library picks (csrc/launch_choice.h), checked on the CPU.

The same header gemm_api.cu compiles is built here with g++ into a small
driver.  Resident-unit counts are those the device query returns on a
152-SM GB300 (76 CTA pairs, 36 four-CTA clusters, 152 single CTAs), passed
in as inputs.  The tests pin the choices for the benchmark shapes and the
rules behind them: the tile width that fills whole waves at the lowest
measured cost per k-block, the 4-CTA multicast unit for rows that are not
a multiple of 128 bytes and only while one GPU is visible, the widths an
MN-major B allows, and when the partial last wave is handed out at run
time.
"""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "dense_gemm_blackwell_persistent_gb300", "csrc")
INCLUDE = os.path.join(ROOT, "include")
SRC = os.path.join(ROOT, "tests", "native", "launch_dump.cpp")
GB300 = (152, 76, 36)   # resident units of 1, 2 and 4 CTAs


@pytest.fixture(scope="module")
def choose(tmp_path_factory):
    exe = str(tmp_path_factory.mktemp("launch") / "launch_dump")
    subprocess.run(["g++", "-O1", "-std=c++17", "-I", CSRC, "-I", INCLUDE, SRC, "-o", exe], check=True)

    def run(M, N, K, ib=2, layout=0, pair=0, mc=-1, visible=1, forced=0, batch=1, mode=-1, capped=0, sk=0,
            resident=GB300):
        line = f"{M} {N} {K} {ib} {layout} {pair} {mc} {visible} {forced} {batch} {mode} {capped} {sk} " \
               f"{resident[0]} {resident[1]} {resident[2]}\n"
        out = subprocess.run([exe], input=line, capture_output=True, text=True, check=True).stdout.split()
        unit, bn, tiles, dyn, units, waves = map(int, out)
        return {"unit": unit, "tile_n": bn, "tiles": tiles, "dynamic": bool(dyn), "units": units, "waves": waves}
    return run


def test_benchmark_shapes(choose):
    # bf16 4096³: 224-wide tiles, 16 × 19 = 304 tiles = 4 whole waves on 76 pairs, static
    assert choose(4096, 4096, 4096) == {"unit": 2, "tile_n": 224, "tiles": 304, "dynamic": False, "units": 0,
                                        "waves": 0}
    # f16 1024×4096×4096: 4 × 19 = 76 tiles, one wave
    r = choose(1024, 4096, 4096)
    assert (r["unit"], r["tile_n"], r["tiles"], r["dynamic"]) == (2, 224, 76, False)
    # bf16 8192³: 256-wide, 1024 tiles = 13 waves + 36 handed out at run time
    r = choose(8192, 8192, 8192)
    assert (r["unit"], r["tile_n"], r["tiles"]) == (2, 256, 1024)
    assert r["dynamic"] and (r["units"], r["waves"]) == (76, 13)
    # ragged 4000×3000×5000: rows of 10 000 bytes -> the 4-CTA multicast unit, 8 × 12 = 96 tiles
    r = choose(4000, 3000, 5000)
    assert (r["unit"], r["tile_n"], r["tiles"], r["dynamic"]) == (4, 256, 96, False)
    # E4M3 4096³: 1-byte elements, rows of 4096 bytes: pairs, 224 wide
    r = choose(4096, 4096, 4096, ib=1)
    assert (r["unit"], r["tile_n"]) == (2, 224)


def test_multicast_needs_one_visible_gpu_and_pairs(choose):
    assert choose(4000, 3000, 5000, visible=2)["unit"] == 2
    assert choose(4000, 3000, 5000, visible=8)["unit"] == 2
    assert choose(4096, 4096, 4096, mc=1)["unit"] == 4
    assert choose(4096, 4096, 4096, mc=1, visible=2)["unit"] == 2     # the run itself is refused by the host
    assert choose(4000, 3000, 5000, mc=0)["unit"] == 2
    assert choose(4000, 3000, 5000, pair=1)["unit"] == 1
    # MN-major operands never multicast by default (their rows run along M or N)
    assert choose(4000, 3000, 5000, layout=2)["unit"] == 2


def test_tile_width_fills_whole_waves(choose):
    """Widest first, a narrower width wins only if its waves × measured
    cycles per k-block are more than 1% cheaper."""
    cycles = {256: 520, 224: 453, 192: 432, 160: 429, 128: 485}
    for M, N, K in [(2048, 2048, 2048), (3072, 3072, 3072), (6144, 6144, 6144), (4096, 8192, 1024),
                    (1000, 776, 1256), (256, 256, 256), (4096, 4096, 4096), (8192, 8192, 8192)]:
        r = choose(M, N, K, pair=2)
        units = {2: 76, 4: 36}[r["unit"]]           # pairs, or the 4-CTA unit for unaligned rows
        tiles_m = -(-M // (128 * r["unit"]))
        best, best_cost = 0, None
        for bn in (256, 224, 192, 160, 128):
            cost = -(-(tiles_m * -(-N // bn)) // units) * cycles[bn]
            if best_cost is None or cost * 100 < best_cost * 99:
                best, best_cost = bn, cost
        assert r["tile_n"] == best, (M, N, K, r)


def test_forced_width_and_mn_major_b(choose):
    assert choose(4096, 4096, 4096, forced=192)["tile_n"] == 192
    # a 4-CTA unit loads a quarter of B's rows: whole 64-element boxes only at width 256
    assert choose(4096, 4096, 4096, layout=2, mc=1)["tile_n"] == 256
    assert choose(4096, 4096, 4096, layout=2, mc=1, forced=224)["tile_n"] == 0
    # pairs take any width with an MN-major B (the padded kernel form)
    assert choose(4096, 4096, 4096, layout=2, forced=224)["tile_n"] == 224


def test_dynamic_list_rules(choose):
    # the partial last wave is handed out from 6 whole waves on (5120³: 400 tiles = 5 whole waves + 20)
    for M in (4096, 5120, 6144, 7168, 8192, 12288):
        r = choose(M, M, M)
        whole, partial = divmod(r["tiles"], 76)
        assert r["dynamic"] == (whole >= 6 and partial > 0), (M, r)
        if r["dynamic"]:
            assert (r["units"], r["waves"]) == (76, whole), (M, r)
    # whole waves only: nothing to hand out
    r = choose(8192, 8192, 8192, forced=256, resident=(152, 64, 36))
    assert r["tiles"] % 64 == 0 and not r["dynamic"]
    # a CTA cap or stream-K keeps the static schedule unless asked for
    assert not choose(8192, 8192, 8192, capped=1)["dynamic"]
    assert not choose(8192, 8192, 8192, sk=1)["dynamic"]
    assert choose(8192, 8192, 8192, capped=1, mode=1)["dynamic"]
    # mode 2: every tile is a list of its own
    r = choose(4096, 4096, 4096, mode=2)
    assert r["dynamic"] and (r["units"], r["waves"]) == (r["tiles"], 1)
    # mode 0: static
    assert not choose(8192, 8192, 8192, mode=0)["dynamic"]


def test_single_ctas_for_small_problems(choose):
    """Left to the library (pair option 0), problems under half a wave of
    256×256 pair tiles whose 128×128 single-CTA tiles fit one wave run on
    single CTAs (a pair's set-up costs more than it saves there); from half
    a wave of pair tiles on, pairs (and the multicast unit where it applies)."""
    assert choose(256, 256, 256)["unit"] == 1                 # 1 pair tile
    assert choose(1024, 1024, 1024)["unit"] == 1              # 16 pair tiles, 64 single tiles
    assert choose(128, 4096, 4096)["unit"] == 1               # 16 pair tiles, 32 single tiles
    assert choose(1000, 776, 1256)["unit"] == 1               # misaligned rows, but small: single CTAs
    assert choose(1024, 4096, 4096)["unit"] == 2              # 64 pair tiles: more than half a wave
    assert choose(1536, 1536, 1024)["unit"] == 1              # 36 pair tiles, 144 single tiles: one wave
    assert choose(1536, 1792, 1024)["unit"] == 2              # 42 pair tiles
    assert choose(1664, 1664, 1024)["unit"] == 2              # 49 pair tiles
    assert choose(1024, 1024, 128, batch=32)["unit"] == 2     # batched: 512 pair tiles
    assert choose(2048, 2048, 2048)["unit"] == 2              # 64 pair tiles
    # an explicit choice or a forced multicast unit is honoured
    assert choose(256, 256, 256, pair=2)["unit"] == 2
    assert choose(1000, 776, 1256, mc=1)["unit"] == 4
    assert choose(4096, 4096, 4096, pair=1)["unit"] == 1


@pytest.fixture(scope="module")
def split(tmp_path_factory):
    exe = str(tmp_path_factory.mktemp("split") / "split_dump")
    subprocess.run(["g++", "-O1", "-std=c++17", "-I", CSRC, "-I", INCLUDE,
                    os.path.join(ROOT, "tests", "native", "split_dump.cpp"), "-o", exe], check=True)

    def run(tiles, units, kb, slice_floats, forced=-1, ws=152 * 4 * 8192):
        line = f"{forced} {tiles} {units} {kb} {slice_floats} {ws}\n"
        return int(subprocess.run([exe], input=line, capture_output=True, text=True, check=True).stdout)
    return run


def test_split_k_choice(split):
    """K slices: a power of two dividing the k-blocks, at least four k-blocks
    each, every slice's tiles in one wave, the partials within the
    workspace; the count minimising k-blocks per slice + a fixed reduction
    cost, and only where that beats the unsplit K loop by a quarter."""
    assert split(4, 152, 128, 256 * 256) == 32          # 256×256×8192 on single CTAs: 4 k-blocks per slice
    assert split(32, 152, 64, 128 * 4096) == 4          # 128×4096×4096: 32 tiles, 4 slices fill the wave
    assert split(9, 152, 64, 384 * 384) == 16           # 384×384×4096
    assert split(76, 76, 64, 1024 * 4096) == 1          # a full wave of tiles already
    assert split(4, 152, 4, 256 * 256) == 1             # 256³: four k-blocks in all
    assert split(64, 152, 16, 1024 * 1024) == 1         # 1024³: a split saves too little
    assert split(4, 152, 128, 4096 * 4096) == 1         # the partials would not fit the workspace
    assert split(4, 152, 100, 65536) == 4               # 100 k-blocks: 4 divides, 8 does not
    assert split(4, 152, 128, 65536, forced=0) == 1     # off
    assert split(4, 152, 128, 65536, forced=8) == 8     # asked for
    assert split(40, 152, 128, 65536, forced=8) == 1    # 320 slices' tiles would not fit one wave


def test_group_height_rule(tmp_path):
    """Raster group height left to the library: every tile row when A is at
    most 48 MB (4096³ bf16: 32 MB, 16 rows of pairs), else 8; never more
    than the tile rows; a forced height is kept (clipped to the tile rows)."""
    src = tmp_path / "group_dump.cpp"
    src.write_text('#include <cstdio>\n#include "launch_choice.h"\nint main(){long long f,t,a;'
                   'while(std::scanf("%lld %lld %lld",&f,&t,&a)==3)std::printf("%d\\n",'
                   'gb300::launch_group_m((int)f,t,a));}\n')
    exe = str(tmp_path / "group_dump")
    subprocess.run(["g++", "-O1", "-std=c++17", "-I", CSRC, "-I", INCLUDE, str(src), "-o", exe], check=True)

    def group(forced, tiles_m, a_bytes):
        out = subprocess.run([exe], input=f"{forced} {tiles_m} {a_bytes}\n", capture_output=True, text=True,
                             check=True).stdout
        return int(out)
    assert group(0, 16, 4096 * 4096 * 2) == 16       # bf16 4096³
    assert group(0, 32, 8192 * 8192 * 2) == 8        # bf16 8192³
    assert group(0, 4, 1024 * 4096 * 2) == 4         # the one-wave shape: its 4 rows
    assert group(0, 8, 4000 * 5000 * 2) == 8         # ragged, 4-CTA units: 40 MB, all 8 rows
    assert group(0, 3, 10 ** 9) == 3                 # never more than the tile rows
    assert group(4, 16, 4096 * 4096 * 2) == 4        # forced
    assert group(64, 16, 10 ** 9) == 16
