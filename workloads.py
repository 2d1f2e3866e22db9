"""Seeded synthetic inputs for the dense GEMM C = A·Bᵀ.

This module only draws numbers: it holds no part of the multiply itself, so
both the CUDA path and the CPU oracle can take their inputs from it without
sharing any arithmetic of the method.

Workloads follow the shapes the pages measure on:
  * bf16 4096³, the single shape the whole series in "Optimizing Blackwell
    Matrix Multiplication in Mojo (Part 2)" is benchmarked on (intro,
    "Starting from a 4-line kernel"); B is stored transposed, N×K.
  * f16 M=1024, K=4096, N=4096, the per-device local matmul of
    "Collective matrix multiplication" (results paragraph).
  * a ragged shape that is a multiple of no tile, the case the masked matmul
    of "Chapter 7: Writing Custom Kernels with Pallas", §4.3 exists for.
  * a small 256³ case and an 8192³ case.
  * bf16 4096³'s shape with 8-bit float inputs (E4M3, bf16 out): the
    float8_e4m3fn operand type of "Writing Mosaic GPU kernels with Pallas",
    "Blackwell (tcgen05)", "Issuing the operation".

Recipe (one reading, stated once): a CPU ``torch.Generator`` seeded with the
workload's seed draws A first, then B, in float32 (``randn`` for normal,
``rand`` scaled to [lo, hi) for uniform, ``randint`` for integers), and torch
casts to bf16/f16 with round-to-nearest-even.  "N(0, 1/sqrt(K))" is read as
standard deviation 1/sqrt(K).  "integers uniform in [-4, 4]" is read as the
nine integers -4..4 inclusive.  8-bit float inputs are drawn the same way
and cast by torch to float8_e4m3fn / float8_e5m2 (nearest, ties to even;
N(0,1) stays far inside both ranges).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

BF16, F16, F32, E4M3, E5M2 = 0, 1, 2, 3, 4   # dtype codes shared with the C ABI's gemm_dtype_t
FP8 = (E4M3, E5M2)
DTYPE_NAMES = {BF16: "bf16", F16: "f16", F32: "f32", E4M3: "e4m3", E5M2: "e5m2"}
TORCH_DTYPES = {BF16: torch.bfloat16, F16: torch.float16, F32: torch.float32,
                E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}
ELEM_BYTES = {BF16: 2, F16: 2, F32: 4, E4M3: 1, E5M2: 1}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dtype: int          # input dtype of A and B
    out_dtype: int      # dtype of C
    dist: str           # "normal", "uniform", "int"
    seed: int
    std: float = 1.0    # for "normal"
    lo: float = -1.0    # for "uniform" / "int" (inclusive bounds for "int")
    hi: float = 1.0

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def compulsory_bytes(self) -> int:
        """Bytes every implementation must move at least once: A, B read, C written."""
        ib, ob = ELEM_BYTES[self.dtype], ELEM_BYTES[self.out_dtype]
        return (self.M * self.K + self.N * self.K) * ib + self.M * self.N * ob

    def describe(self) -> str:
        d = {"normal": f"N(0,{self.std:g})", "uniform": f"U({self.lo:g},{self.hi:g})",
             "int": f"int[{int(self.lo)},{int(self.hi)}]"}[self.dist]
        return (f"{self.name}: M={self.M} N={self.N} K={self.K} {DTYPE_NAMES[self.dtype]} in, "
                f"{DTYPE_NAMES[self.out_dtype]} out, {d}, seed {self.seed}")


WORKLOADS = {
    "gemm_256_f32out": Workload("gemm_256_f32out", 256, 256, 256, BF16, F32, "normal", 0),
    "gemm_256_int": Workload("gemm_256_int", 256, 256, 256, BF16, F32, "int", 0, lo=-4, hi=4),
    "gemm_4096_bf16": Workload("gemm_4096_bf16", 4096, 4096, 4096, BF16, BF16, "normal", 1),
    "gemm_1024x4096x4096_f16": Workload("gemm_1024x4096x4096_f16", 1024, 4096, 4096, F16, F16, "normal", 2),
    "gemm_ragged_4000x3000x5000": Workload("gemm_ragged_4000x3000x5000", 4000, 3000, 5000, BF16, F32,
                                           "uniform", 3, lo=-1.0, hi=1.0),
    "gemm_8192_bf16": Workload("gemm_8192_bf16", 8192, 8192, 8192, BF16, BF16, "normal", 4,
                               std=1.0 / math.sqrt(8192)),
    "gemm_4096_e4m3": Workload("gemm_4096_e4m3", 4096, 4096, 4096, E4M3, BF16, "normal", 5),
}


def _draw(gen: torch.Generator, rows: int, cols: int, w: Workload) -> torch.Tensor:
    if w.dist == "normal":
        x = torch.randn(rows, cols, generator=gen, dtype=torch.float32)
        if w.std != 1.0:
            x.mul_(w.std)
    elif w.dist == "uniform":
        x = torch.rand(rows, cols, generator=gen, dtype=torch.float32)
        x.mul_(w.hi - w.lo).add_(w.lo)
    elif w.dist == "int":
        x = torch.randint(int(w.lo), int(w.hi) + 1, (rows, cols), generator=gen).to(torch.float32)
    else:
        raise ValueError(f"unknown distribution {w.dist!r}")
    return x.to(TORCH_DTYPES[w.dtype])


def make_inputs(w: Workload, M: Optional[int] = None, N: Optional[int] = None,
                K: Optional[int] = None, seed: Optional[int] = None):
    """Return CPU tensors (A [M,K], B [N,K]) in the workload's input dtype.

    Shape and seed may be overridden to draw a smaller case with the same
    distribution (used by parity sweeps over many shapes).
    """
    M = w.M if M is None else M
    N = w.N if N is None else N
    K = w.K if K is None else K
    gen = torch.Generator(device="cpu")
    gen.manual_seed(w.seed if seed is None else seed)
    A = _draw(gen, M, K, w)
    B = _draw(gen, N, K, w)
    return A.contiguous(), B.contiguous()


def as_bits(t: torch.Tensor) -> np.ndarray:
    """The raw bit patterns of a CPU input tensor: uint16 for bf16/f16, uint8 for fp8."""
    if t.dtype in (torch.float8_e4m3fn, torch.float8_e5m2):
        return t.contiguous().view(torch.uint8).numpy()
    assert t.dtype in (torch.bfloat16, torch.float16)
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def workload_by_name(name: str) -> Workload:
    return WORKLOADS[name]
