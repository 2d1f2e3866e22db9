"""CPU oracle for C = A·Bᵀ (fp64), with its build step.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg and reference arm (``--impl reference``) are the
only callers.  The library's product path
never imports this package, and this package imports nothing from the library.

The arithmetic lives in ``gemm_oracle.c`` (plain C, fp64 triple loop,
OpenMP over rows); this module compiles it with gcc and wraps it with ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libgemm_oracle.so")
_lock = threading.Lock()

BF16, F16, F32, E4M3, E5M2 = 0, 1, 2, 3, 4
FP8 = (E4M3, E5M2)


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle into ``oracle/_build/libgemm_oracle.so`` (gcc, OpenMP).

    ``src``/``out`` let a test compile a copy of the source elsewhere."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(path: str):
    lib = ctypes.CDLL(path)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    dp = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    lib.oracle_decode16.restype = ctypes.c_double
    lib.oracle_decode16.argtypes = [ctypes.c_uint16, ctypes.c_int]
    lib.oracle_encode16.restype = ctypes.c_uint16
    lib.oracle_encode16.argtypes = [ctypes.c_double, ctypes.c_int]
    lib.oracle_decode16_array.restype = None
    lib.oracle_decode16_array.argtypes = [u16p, dp, ctypes.c_int64, ctypes.c_int]
    lib.oracle_encode16_array.restype = None
    lib.oracle_encode16_array.argtypes = [dp, u16p, ctypes.c_int64, ctypes.c_int]
    u8p = ctypes.POINTER(ctypes.c_uint8)
    lib.oracle_decode8.restype = ctypes.c_double
    lib.oracle_decode8.argtypes = [ctypes.c_uint8, ctypes.c_int]
    lib.oracle_decode8_array.restype = None
    lib.oracle_decode8_array.argtypes = [u8p, dp, ctypes.c_int64, ctypes.c_int]
    vp = ctypes.c_void_p
    lib.oracle_gemm.restype = ctypes.c_int
    lib.oracle_gemm.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                ctypes.c_int64, dp, dp, ctypes.c_int]
    lib.oracle_gemm_entries.restype = ctypes.c_int
    lib.oracle_gemm_entries.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int64,
                                        ctypes.c_int64, ctypes.c_int64, i64p, i64p,
                                        ctypes.c_int64, dp, dp, ctypes.c_int]
    lib.oracle_max_threads.restype = ctypes.c_int
    lib.oracle_max_threads.argtypes = []
    return lib


def _u16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16:
        raise TypeError("expected the raw 16-bit patterns as a uint16 array")
    return x


def _in_bits(x: np.ndarray, dtype: int) -> np.ndarray:
    """Input patterns: uint16 for bf16/f16, uint8 for the fp8 formats."""
    x = np.ascontiguousarray(x)
    want = np.uint8 if dtype in FP8 else np.uint16
    if x.dtype != want:
        raise TypeError(f"expected the raw bit patterns as a {np.dtype(want).name} array for dtype {dtype}")
    return x


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


class Oracle:
    """ctypes view of one compiled copy of ``gemm_oracle.c``."""

    def __init__(self, path: str):
        self.path = path
        self.lib = _bind(path)

    def decode(self, bits: np.ndarray, dtype: int) -> np.ndarray:
        """Exact float64 values of bf16 (0), f16 (1), E4M3 (3) or E5M2 (4) bit patterns."""
        bits = _in_bits(bits, dtype)
        out = np.empty(bits.shape, dtype=np.float64)
        if dtype in FP8:
            self.lib.oracle_decode8_array(_ptr(bits, ctypes.c_uint8), _ptr(out, ctypes.c_double),
                                          bits.size, dtype)
        else:
            self.lib.oracle_decode16_array(_ptr(bits, ctypes.c_uint16), _ptr(out, ctypes.c_double),
                                           bits.size, dtype)
        return out

    def encode(self, x: np.ndarray, dtype: int) -> np.ndarray:
        """Round float64 values to bf16/f16 (nearest, ties to even); returns bit patterns."""
        x = np.ascontiguousarray(x, dtype=np.float64)
        out = np.empty(x.shape, dtype=np.uint16)
        self.lib.oracle_encode16_array(_ptr(x, ctypes.c_double), _ptr(out, ctypes.c_uint16),
                                       x.size, dtype)
        return out

    def gemm(self, A_bits: np.ndarray, B_bits: np.ndarray, dtype: int, threads: int = 0
             ) -> Tuple[np.ndarray, np.ndarray]:
        """C = A·Bᵀ and S = |A|·|B|ᵀ in float64.  A: [M,K], B: [N,K] bit patterns."""
        A_bits, B_bits = _in_bits(A_bits, dtype), _in_bits(B_bits, dtype)
        if A_bits.ndim != 2 or B_bits.ndim != 2 or A_bits.shape[1] != B_bits.shape[1]:
            raise ValueError("A must be [M,K] and B [N,K]")
        M, K = A_bits.shape
        N = B_bits.shape[0]
        C = np.zeros((M, N), dtype=np.float64)
        S = np.zeros((M, N), dtype=np.float64)
        rc = self.lib.oracle_gemm(A_bits.ctypes.data, B_bits.ctypes.data,
                                  dtype, M, N, K, _ptr(C, ctypes.c_double),
                                  _ptr(S, ctypes.c_double), threads)
        if rc != 0:
            raise RuntimeError(f"oracle_gemm failed ({rc})")
        return C, S

    def gemm_entries(self, A_bits: np.ndarray, B_bits: np.ndarray, dtype: int, I: np.ndarray,
                     J: np.ndarray, threads: int = 0) -> Tuple[np.ndarray, np.ndarray]:
        """C[I[t], J[t]] and S[I[t], J[t]] only, for sampled checks of large outputs."""
        A_bits, B_bits = _in_bits(A_bits, dtype), _in_bits(B_bits, dtype)
        M, K = A_bits.shape
        N = B_bits.shape[0]
        I = np.ascontiguousarray(I, dtype=np.int64)
        J = np.ascontiguousarray(J, dtype=np.int64)
        if I.shape != J.shape:
            raise ValueError("I and J must have the same shape")
        C = np.zeros(I.shape, dtype=np.float64)
        S = np.zeros(I.shape, dtype=np.float64)
        rc = self.lib.oracle_gemm_entries(A_bits.ctypes.data, B_bits.ctypes.data, dtype, M, N, K,
                                          _ptr(I, ctypes.c_int64), _ptr(J, ctypes.c_int64),
                                          I.size, _ptr(C, ctypes.c_double),
                                          _ptr(S, ctypes.c_double), threads)
        if rc != 0:
            raise RuntimeError(f"oracle_gemm_entries failed ({rc})")
        return C, S

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())


_default: Optional[Oracle] = None


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def decode(bits, dtype):
    return default().decode(bits, dtype)


def encode(x, dtype):
    return default().encode(x, dtype)


def gemm(A_bits, B_bits, dtype, threads: int = 0):
    return default().gemm(A_bits, B_bits, dtype, threads)


def gemm_entries(A_bits, B_bits, dtype, I, J, threads: int = 0):
    return default().gemm_entries(A_bits, B_bits, dtype, I, J, threads)


def max_threads() -> int:
    return default().max_threads()


SOURCE = _SRC
