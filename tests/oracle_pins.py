"""Pins for the CPU oracle: checks against facts fixed outside the oracle.

Each pin takes an ``oracle.Oracle`` and raises AssertionError when the oracle
disagrees with what the number formats, the mathematics or an independent
library routine fix.  They are run on the real oracle (all must pass) and on
copies with planted mistakes (each copy must fail at least one).

What pins what:
  * decode/encode of the 16-bit formats: a hand-derived bit-pattern table
    (tests/golden), every one of the 65536 patterns against numpy's binary16
    and torch's bfloat16, and rounding against those libraries' conversions.
  * decode of the 8-bit float formats (E4M3 "fn" and E5M2): a hand-derived
    table (tests/golden) and every one of the 256 patterns of each against
    torch's float8 types.
  * the product: a hand-worked example (tests/golden), closed forms (identity,
    all-ones, rank-1 outer products with distinct factors), exact rational
    brute force on every shape up to 8×8×8 for the 16-bit formats (up to
    4×4×4 for the 8-bit ones), numpy float64 matmul within the
    float64 summation bound, symmetry C(B,A) = C(A,B)ᵀ, power-of-two
    scaling, IEEE special values, and empty sizes; for fp8 inputs, exact
    rational brute force, agreement with the bf16 path on values both
    formats hold, and sampled entries against the exact sum.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np
import torch

BF16, F16, E4M3, E5M2 = 0, 1, 3, 4
FP8_TORCH = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _bits_of(x: np.ndarray, dtype: int) -> np.ndarray:
    """Bit patterns of values exactly representable in the 16-bit format (library cast)."""
    t = torch.tensor(np.asarray(x, dtype=np.float32), dtype=torch.float32)
    t = t.to(torch.bfloat16 if dtype == BF16 else torch.float16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _rand_bits(rng: np.random.Generator, shape, dtype: int, scale: float = 1.0) -> np.ndarray:
    return _bits_of(rng.standard_normal(shape) * scale, dtype)


def _fp8_bits_of(x: np.ndarray, dtype: int) -> np.ndarray:
    """fp8 patterns of values (library cast, round to nearest even)."""
    t = torch.tensor(np.asarray(x, dtype=np.float32), dtype=torch.float32).to(FP8_TORCH[dtype])
    return t.view(torch.uint8).numpy().copy()


def _fp8_finite_random(rng: np.random.Generator, shape, dtype: int) -> np.ndarray:
    """Uniformly random finite fp8 patterns: every exponent, subnormals and zeros included."""
    bits = rng.integers(0, 256, size=shape, dtype=np.int64).astype(np.uint8)
    if dtype == E4M3:
        bad = (bits & 0x7F) == 0x7F
    else:
        bad = (bits & 0x7C) == 0x7C
    bits[bad] = 0x00
    return bits


# ---------------------------------------------------------------- formats

def pin_decode_golden(o):
    path = os.path.join(GOLDEN, "float16_bfloat16_bits.txt")
    n = 0
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, hexbits, value = line.split()[:3]
        dt = BF16 if name == "bf16" else F16
        got = o.decode(np.array([int(hexbits, 16)], dtype=np.uint16), dt)[0]
        want = float(value)
        assert got == want and np.signbit(got) == np.signbit(want), (name, hexbits, got, want)
        n += 1
    assert n >= 20


def pin_decode_all_f16_vs_numpy(o):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = o.decode(bits, F16)
    with np.errstate(invalid="ignore"):   # the NaN patterns cast to NaN, as wanted
        want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def pin_decode_all_bf16_vs_torch(o):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = o.decode(bits, BF16)
    want = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def pin_decode_fp8_golden(o):
    path = os.path.join(GOLDEN, "float8_bits.txt")
    n = 0
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, hexbits, value = line.split()[:3]
        dt = E4M3 if name == "e4m3" else E5M2
        got = o.decode(np.array([int(hexbits, 16)], dtype=np.uint8), dt)[0]
        want = float(value)
        if np.isnan(want):
            assert np.isnan(got), (name, hexbits, got)
        else:
            assert got == want and np.signbit(got) == np.signbit(want), (name, hexbits, got, want)
        n += 1
    assert n >= 20


def pin_decode_all_fp8_vs_torch(o):
    bits = np.arange(256, dtype=np.uint32).astype(np.uint8)
    for dt, tdt in FP8_TORCH.items():
        got = o.decode(bits, dt)
        want = torch.from_numpy(bits.copy()).view(tdt).to(torch.float64).numpy()
        nan = np.isnan(want)
        assert np.array_equal(np.isnan(got), nan), dt
        assert np.array_equal(got[~nan], want[~nan]), dt
        assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan])), dt


def _encode_probe_values(rng, dtype):
    """Random values, exact midpoints between neighbours (ties), subnormals, overflow edge."""
    bits = rng.integers(0, 65536, size=20000).astype(np.uint16)
    if dtype == F16:
        with np.errstate(invalid="ignore"):   # NaN patterns among the random bits
            vals = bits.view(np.float16).astype(np.float64)
            nxt = np.nextafter(bits.view(np.float16), np.float16(np.inf)).astype(np.float64)
    else:
        vals = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
        nb = (bits.astype(np.int32) + np.where(bits < 0x8000, 1, -1)).astype(np.uint16)
        nxt = torch.from_numpy(nb.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    ok = np.isfinite(vals) & np.isfinite(nxt)
    mids = (vals[ok] + nxt[ok]) / 2.0                       # exact ties
    rnd = rng.standard_normal(20000) * np.exp2(rng.integers(-30, 20, size=20000))
    sub = rng.standard_normal(2000) * (2.0 ** -24 if dtype == F16 else 2.0 ** -130)
    big = np.array([65504.0, 65519.99, 65520.0, 65536.0, 1e6, -65520.0])
    return np.concatenate([vals[ok], mids, rnd, sub, big, [0.0, -0.0]])


def pin_encode_vs_numpy_f16(o):
    rng = np.random.default_rng(11)
    x = _encode_probe_values(rng, F16)
    got = o.encode(x, F16)
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)         # numpy rounds double -> half once
    assert np.array_equal(got, want), int((got != want).sum())


def pin_encode_vs_torch_bf16(o):
    rng = np.random.default_rng(12)
    x = _encode_probe_values(rng, BF16)
    x = x[np.abs(x) < 3.0e38]
    x32 = x.astype(np.float32)
    x = x[x32.astype(np.float64) == x]                      # only values exact in float32: one rounding
    got = o.encode(x, BF16)
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want), int((got != want).sum())


# ---------------------------------------------------------------- product

def _read_worked():
    rows = {"A": [], "B": [], "C": [], "S": []}
    dims = {}
    for line in open(os.path.join(GOLDEN, "gemm_worked_2x2x3.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        if key in dims or key in ("M", "N", "K"):
            dims[key] = int(vals[0])
        else:
            rows[key].append([float(v) for v in vals])
    return dims, {k: np.array(v) for k, v in rows.items()}


def pin_worked_example(o):
    dims, r = _read_worked()
    for dt in (BF16, F16):
        C, S = o.gemm(_bits_of(r["A"], dt), _bits_of(r["B"], dt), dt)
        assert C.shape == (dims["M"], dims["N"])
        assert np.array_equal(C, r["C"]), (dt, C)
        assert np.array_equal(S, r["S"]), (dt, S)


def pin_identity(o):
    rng = np.random.default_rng(1)
    K, N = 12, 7                                            # A = I (M = K), B: N×K, non-square
    for dt in (BF16, F16):
        A = _bits_of(np.eye(K), dt)
        B = _rand_bits(rng, (N, K), dt)
        C, _ = o.gemm(A, B, dt)
        assert C.shape == (K, N)
        assert np.array_equal(C, o.decode(B, dt).T)


def pin_all_ones(o):
    for (M, N, K) in [(1, 1, 1), (5, 3, 7), (33, 17, 129), (13, 9, 1000)]:
        for dt in (BF16, F16):
            A = _bits_of(np.ones((M, K)), dt)
            B = _bits_of(np.ones((N, K)), dt)
            C, S = o.gemm(A, B, dt)
            assert np.all(C == K) and np.all(S == K), (M, N, K)


def pin_rank1(o):
    # a(i,k) = u_i x_k, b(j,k) = v_j y_k  =>  C[i,j] = u_i v_j sum_k x_k y_k, exactly.
    rng = np.random.default_rng(2)
    M, N, K = 6, 5, 9
    u = rng.integers(-4, 5, M).astype(np.float64)
    v = rng.integers(-4, 5, N).astype(np.float64)
    x = rng.integers(-3, 4, K).astype(np.float64)
    y = rng.integers(1, 4, K).astype(np.float64)
    for dt in (BF16, F16):
        A = _bits_of(np.outer(u, x), dt)
        B = _bits_of(np.outer(v, y), dt)
        C, S = o.gemm(A, B, dt)
        assert np.array_equal(C, np.outer(u, v) * float(np.dot(x, y)))
        assert np.array_equal(S, np.outer(np.abs(u), np.abs(v)) * float(np.dot(np.abs(x), np.abs(y))))


def pin_bruteforce_exact(o):
    # Every shape 1..8 in each of M, N, K (512 shapes): the exact rational sum,
    # rounded once, must equal the oracle (fp64 sums of up to eight products
    # of these N(0,1)-drawn bf16/f16 values are exact).
    rng = np.random.default_rng(3)
    for dt in (BF16, F16):
        for M in range(1, 9):
            for N in range(1, 9):
                for K in range(1, 9):
                    A = _rand_bits(rng, (M, K), dt)
                    B = _rand_bits(rng, (N, K), dt)
                    a, b = o.decode(A, dt), o.decode(B, dt)
                    C, S = o.gemm(A, B, dt)
                    for i in range(M):
                        for j in range(N):
                            exact = sum((Fraction(a[i, k]) * Fraction(b[j, k]) for k in range(K)),
                                        Fraction(0))
                            mag = sum((abs(Fraction(a[i, k]) * Fraction(b[j, k])) for k in range(K)),
                                      Fraction(0))
                            assert C[i, j] == float(exact), (dt, M, N, K, i, j)
                            assert S[i, j] == float(mag), (dt, M, N, K, i, j)


def pin_numpy_float64(o):
    # M=100, K=200, N=130: the non-divisible shape of the masked matmul in
    # "Chapter 7: Writing Custom Kernels with Pallas", §4.3.
    rng = np.random.default_rng(4)
    M, K, N = 100, 200, 130
    for dt in (BF16, F16):
        A = _rand_bits(rng, (M, K), dt)
        B = _rand_bits(rng, (N, K), dt)
        C, S = o.gemm(A, B, dt)
        ref = o.decode(A, dt) @ o.decode(B, dt).T
        bound = 2.0 * K * 2.0 ** -53 * S
        assert np.all(np.abs(C - ref) <= bound)
        ref_abs = np.abs(o.decode(A, dt)) @ np.abs(o.decode(B, dt)).T
        assert np.all(np.abs(S - ref_abs) <= bound)


def pin_swap_symmetry(o):
    rng = np.random.default_rng(5)
    A = _rand_bits(rng, (19, 37), BF16)
    B = _rand_bits(rng, (23, 37), BF16)
    C1, S1 = o.gemm(A, B, BF16)
    C2, S2 = o.gemm(B, A, BF16)
    assert np.array_equal(C1, C2.T) and np.array_equal(S1, S2.T)


def pin_power_of_two_scaling(o):
    rng = np.random.default_rng(6)
    x = rng.standard_normal((11, 29))
    A1, A2 = _bits_of(x, BF16), _bits_of(4.0 * x, BF16)     # x4 is exact in bf16
    B = _rand_bits(rng, (8, 29), BF16)
    C1, _ = o.gemm(A1, B, BF16)
    C2, _ = o.gemm(A2, B, BF16)
    assert np.array_equal(C2, 4.0 * C1)


def pin_linearity_in_a(o):
    # C(A1 + A2, B) = C(A1, B) + C(A2, B): small integers, so every operand,
    # product and sum is exact in bf16/fp64 and the identity holds bit for bit.
    rng = np.random.default_rng(7)
    x1 = rng.integers(-8, 9, size=(13, 41)).astype(np.float64)
    x2 = rng.integers(-8, 9, size=(13, 41)).astype(np.float64)
    B = _bits_of(rng.integers(-8, 9, size=(17, 41)), BF16)
    C1, _ = o.gemm(_bits_of(x1, BF16), B, BF16)
    C2, _ = o.gemm(_bits_of(x2, BF16), B, BF16)
    C12, _ = o.gemm(_bits_of(x1 + x2, BF16), B, BF16)
    assert np.array_equal(C12, C1 + C2)
    assert np.abs(C1).max() > 0 and not np.array_equal(C1, C2)


def pin_special_values(o):
    # IEEE: inf·positive = inf, inf·0 = NaN, NaN propagates.
    A = _bits_of(np.array([[np.inf, 1.0], [1.0, np.nan], [1.0, 1.0]]), BF16)
    B = _bits_of(np.array([[2.0, 3.0], [0.0, 1.0]]), BF16)
    C, _ = o.gemm(A, B, BF16)
    assert C[0, 0] == np.inf and np.isnan(C[0, 1])
    assert np.isnan(C[1, 0]) and np.isnan(C[1, 1])
    assert C[2, 0] == 5.0 and C[2, 1] == 1.0


def pin_empty_sizes(o):
    C, S = o.gemm(np.zeros((3, 0), np.uint16), np.zeros((4, 0), np.uint16), BF16)
    assert C.shape == (3, 4) and np.all(C == 0) and np.all(S == 0)       # empty sum
    C, _ = o.gemm(np.zeros((0, 5), np.uint16), np.zeros((4, 5), np.uint16), BF16)
    assert C.shape == (0, 4)


def pin_entries_agree(o):
    # Sampled entries: same definition; compared with the exact rational sum.
    rng = np.random.default_rng(7)
    M, N, K = 37, 41, 53
    A = _rand_bits(rng, (M, K), F16)
    B = _rand_bits(rng, (N, K), F16)
    I = rng.integers(0, M, 60)
    J = rng.integers(0, N, 60)
    C, S = o.gemm_entries(A, B, F16, I, J)
    a, b = o.decode(A, F16), o.decode(B, F16)
    for t in range(60):
        exact = sum((Fraction(a[I[t], k]) * Fraction(b[J[t], k]) for k in range(K)), Fraction(0))
        assert abs(C[t] - float(exact)) <= 2.0 * K * 2.0 ** -53 * S[t]
        assert S[t] >= abs(C[t])


def pin_fp8_bruteforce(o):
    # Every shape 1..4 in M, N, K on random finite fp8 patterns (all exponents,
    # subnormals): the oracle is within the sequential fp64 summation bound of
    # the exact rational sum, and S is the exact magnitude sum rounded within
    # the same bound.  On values cast from N(0,1) (a narrow exponent range) the
    # fp64 sums are exact and must match the rational sum exactly.
    rng = np.random.default_rng(11)
    for dt in (E4M3, E5M2):
        for M in range(1, 5):
            for N in range(1, 5):
                for K in range(1, 5):
                    for gen in ("wide", "narrow"):
                        if gen == "wide":
                            A, B = _fp8_finite_random(rng, (M, K), dt), _fp8_finite_random(rng, (N, K), dt)
                        else:
                            A = _fp8_bits_of(rng.standard_normal((M, K)), dt)
                            B = _fp8_bits_of(rng.standard_normal((N, K)), dt)
                        a, b = o.decode(A, dt), o.decode(B, dt)
                        C, S = o.gemm(A, B, dt)
                        for i in range(M):
                            for j in range(N):
                                prods = [Fraction(a[i, k]) * Fraction(b[j, k]) for k in range(K)]
                                exact, mag = sum(prods, Fraction(0)), sum((abs(p) for p in prods), Fraction(0))
                                if gen == "narrow":
                                    assert C[i, j] == float(exact) and S[i, j] == float(mag), (dt, M, N, K)
                                else:
                                    bound = 2.0 * K * 2.0 ** -53 * float(mag)
                                    assert abs(C[i, j] - float(exact)) <= bound, (dt, M, N, K, i, j)
                                    assert abs(S[i, j] - float(mag)) <= bound, (dt, M, N, K, i, j)


def pin_fp8_matches_bf16_on_shared_values(o):
    # Values held exactly by both fp8 formats and by bf16 (small integers and
    # halves): the same sums whichever format carries them.
    rng = np.random.default_rng(12)
    x = rng.integers(-8, 9, size=(23, 45)) / 2.0
    y = rng.integers(-8, 9, size=(17, 45)) / 2.0
    C16, S16 = o.gemm(_bits_of(x, BF16), _bits_of(y, BF16), BF16)
    for dt in (E4M3, E5M2):
        C8, S8 = o.gemm(_fp8_bits_of(x, dt), _fp8_bits_of(y, dt), dt)
        assert np.array_equal(C8, C16) and np.array_equal(S8, S16), dt
        assert np.array_equal(C8, x @ y.T)


def pin_fp8_entries_agree(o):
    rng = np.random.default_rng(13)
    M, N, K = 29, 31, 41
    for dt in (E4M3, E5M2):
        A = _fp8_bits_of(rng.standard_normal((M, K)), dt)
        B = _fp8_bits_of(rng.standard_normal((N, K)), dt)
        I = rng.integers(0, M, 50)
        J = rng.integers(0, N, 50)
        C, S = o.gemm_entries(A, B, dt, I, J)
        a, b = o.decode(A, dt), o.decode(B, dt)
        for t in range(50):
            exact = sum((Fraction(a[I[t], k]) * Fraction(b[J[t], k]) for k in range(K)), Fraction(0))
            assert C[t] == float(exact), (dt, t)
            assert S[t] >= abs(C[t])


ALL_PINS = [
    pin_decode_golden, pin_decode_all_f16_vs_numpy, pin_decode_all_bf16_vs_torch,
    pin_encode_vs_numpy_f16, pin_encode_vs_torch_bf16, pin_worked_example, pin_identity,
    pin_all_ones, pin_rank1, pin_bruteforce_exact, pin_numpy_float64, pin_swap_symmetry,
    pin_power_of_two_scaling, pin_linearity_in_a, pin_special_values, pin_empty_sizes, pin_entries_agree,
    pin_decode_fp8_golden, pin_decode_all_fp8_vs_torch, pin_fp8_bruteforce,
    pin_fp8_matches_bf16_on_shared_values, pin_fp8_entries_agree,
]
