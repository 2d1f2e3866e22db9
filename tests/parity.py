"""Comparison helpers shared by the GPU parity tests.

The tolerance is the one stated for this GEMM (bf16/f16 in, fp32 accumulate):
  fp32 output:      |C - C_ref| <= 1e-5 * S
  bf16/f16 output:  |C - C_ref| <= 2^-8 * |C_ref| + 1e-5 * S
where C_ref is the fp64 oracle and S = sum_k |a_ik| |b_jk| (also from the
oracle).  1e-5·S bounds fp32 accumulation in any order; 2^-8·|C_ref| is one
rounding to bf16, whose unit the pages give as about 2^-8 ("Chapter 7:
Writing Custom Kernels with Pallas", §4.1').  On small-integer inputs every
partial sum is exact, so the bar there is equality (fp32 out) or equality
with the oracle's round-to-nearest-even of the exact sum (16-bit out).
"""
from __future__ import annotations

import numpy as np
import torch

import workloads as wl

REL_16BIT = 2.0 ** -8
ABS_ACC = 1e-5


def to_f64(C: torch.Tensor) -> np.ndarray:
    return C.detach().to("cpu", torch.float64).numpy()


def tolerance(C_ref: np.ndarray, S: np.ndarray, out_dtype: int) -> np.ndarray:
    tol = ABS_ACC * S
    if out_dtype in (wl.BF16, wl.F16):
        tol = tol + REL_16BIT * np.abs(C_ref)
    return tol


def assert_within(C: np.ndarray, C_ref: np.ndarray, S: np.ndarray, out_dtype: int, what: str = ""):
    assert C.shape == C_ref.shape, (C.shape, C_ref.shape)
    err = np.abs(C - C_ref)
    tol = tolerance(C_ref, S, out_dtype)
    bad = ~(err <= tol)                         # NaN counts as bad
    if bad.any():
        idx = np.argwhere(bad)
        first = tuple(idx[0])
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.size} elements out of tolerance; first at {first}: "
            f"got {C[first]!r}, want {C_ref[first]!r}, tol {tol[first]!r}; "
            f"max err/tol {float(np.nanmax(np.where(tol > 0, err / np.maximum(tol, 1e-300), err))):.3g}")


def sample_positions(M: int, N: int, n_random: int, seed: int, tile_m: int = 128, tile_n: int = 256):
    """Corners, tile edges and the ragged tail, plus uniform random positions."""
    rng = np.random.default_rng(seed)
    rows = {0, 1, M - 1, M - 2}
    cols = {0, 1, N - 1, N - 2}
    for r in range(tile_m, M, tile_m):
        rows.update((r - 1, r))
    for c in range(tile_n, N, tile_n):
        cols.update((c - 1, c))
    rows = np.array(sorted(x for x in rows if 0 <= x < M))
    cols = np.array(sorted(x for x in cols if 0 <= x < N))
    # edge rows × random columns, random rows × edge columns, then uniform
    I = [np.repeat(rows, 4), rng.integers(0, M, cols.size * 4), rng.integers(0, M, n_random)]
    J = [rng.integers(0, N, rows.size * 4), np.repeat(cols, 4), rng.integers(0, N, n_random)]
    I.append(np.array([0, 0, M - 1, M - 1]))
    J.append(np.array([0, N - 1, 0, N - 1]))
    return np.concatenate(I).astype(np.int64), np.concatenate(J).astype(np.int64)
