"""Python binding of the GB300 dense GEMM library (C = A·Bᵀ).

Argument marshalling only: every function forwards to the extern "C" entry
point of the same name in ``_lib/libgb300gemm.so`` (declared in
include/gemm.h).  All arithmetic runs in the library's CUDA kernels.  If the
compiled library is missing, importing this package raises at once: there is
no fallback implementation.

``matmul`` is a convenience for torch tensors: it checks shapes, allocates C
with torch (memory only) and calls ``gemm_plan_run`` on the current stream.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import _build

GEMM_BF16, GEMM_F16, GEMM_F32, GEMM_E4M3, GEMM_E5M2 = 0, 1, 2, 3, 4
GEMM_OK = 0
GEMM_ERR_INVALID_ARG = -1
GEMM_ERR_UNSUPPORTED = -2
GEMM_ERR_MISALIGNED = -3
GEMM_ERR_CUDA = -4
GEMM_ERR_DRIVER = -5
GEMM_ERR_NO_PLAN = -6
GEMM_ERR_TIMEOUT = -7
GEMM_ERR_NO_DEVICE = -8
GEMM_ERR_INTERNAL = -9
GEMM_OPT_CTA_PAIR, GEMM_OPT_GROUP_M, GEMM_OPT_MAX_CTAS, GEMM_OPT_TILE_N, GEMM_OPT_STREAM_K = 1, 2, 3, 4, 5
GEMM_OPT_MULTICAST = 6
GEMM_OPT_WAIT_LIMIT_US = 7
GEMM_OPT_STALL_TEST = 8
GEMM_OPT_DYNAMIC = 9
GEMM_OPT_FAIL_ENCODE = 10
GEMM_OPT_VISIBLE_DEVICES = 11
GEMM_OPT_CLOCK_LOG = 12
GEMM_OPT_PDL = 13
GEMM_OPT_SPLIT_K = 14
GEMM_K_MAJOR, GEMM_A_MN_MAJOR, GEMM_B_MN_MAJOR = 0, 1, 2

# GB300_GEMM_VARIANT=trace selects the GEMM_TRACE build (timeline stamps),
# GB300_GEMM_VARIANT=debug the GEMM_DEBUG build (consistency checks in the kernel).
VARIANT = os.environ.get("GB300_GEMM_VARIANT", "")
LIB_PATH = _build.lib_path(VARIANT)

_REBUILD = ("build the CUDA library first (python dense_gemm_blackwell_persistent_gb300/_build.py, "
            "or __graft_entry__.build())")
if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: {_REBUILD}")

_lib = ctypes.CDLL(LIB_PATH)
_missing = [n for n in ("gemm_plan_create", "gemm_plan_run_batched", "gemm_probe_mma_rate_n", "gemm_run_noalloc",
                        "gemm_plan_clock_log")
            if not hasattr(_lib, n)]
if _missing:
    raise ImportError(f"{LIB_PATH} is out of date (no {', '.join(_missing)}): {_REBUILD}")

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int

_lib.gemm_plan_create.argtypes = [ctypes.POINTER(_vp), _int, ctypes.c_uint]
_lib.gemm_plan_set_option.argtypes = [_vp, _int, _i64]
_lib.gemm_run.argtypes = [_vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _vp]
_lib.gemm_plan_run.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _vp]
_lib.gemm_plan_run_host.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _vp]
_lib.gemm_plan_run_layout.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _int, _vp]
_lib.gemm_plan_run_batched.argtypes = [_vp, _vp, _vp, _vp] + [_i64] * 7 + [_int, _int, _int, _vp]
_lib.gemm_run_noalloc.argtypes = [_vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _vp]
_lib.gemm_plan_status.argtypes = [_vp, ctypes.POINTER(_int)]
_lib.gemm_plan_last_grid.argtypes = [_vp, ctypes.POINTER(_int)]
_lib.gemm_plan_last_tile_n.argtypes = [_vp, ctypes.POINTER(_int)]
_lib.gemm_plan_last_split.argtypes = [_vp, ctypes.POINTER(_int)]
_lib.gemm_plan_last_launch.argtypes = [_vp] + [ctypes.POINTER(_int)] * 5
_lib.gemm_plan_destroy.argtypes = [_vp]
_lib.gemm_plan_trace.argtypes = [_vp, _vp, ctypes.c_size_t, ctypes.POINTER(_int), ctypes.POINTER(_int)]
_lib.gemm_plan_clock_log.argtypes = [_vp, ctypes.POINTER(ctypes.c_uint64), _i64, ctypes.POINTER(_i64)]
_lib.gemm_probe_mma_rate.argtypes = [_int, _int, _i64] + [ctypes.POINTER(ctypes.c_double)] * 3
_lib.gemm_probe_mma_rate_n.argtypes = [_int, _int, _int, _i64] + [ctypes.POINTER(ctypes.c_double)] * 3
_lib.gemm_strerror.argtypes = [_int]
_lib.gemm_strerror.restype = ctypes.c_char_p
for _name in ("gemm_plan_create", "gemm_plan_set_option", "gemm_run", "gemm_run_noalloc", "gemm_plan_run",
              "gemm_plan_run_host", "gemm_plan_run_layout", "gemm_plan_run_batched", "gemm_plan_status", "gemm_plan_last_grid", "gemm_plan_last_tile_n",
              "gemm_plan_last_launch", "gemm_plan_last_split",
              "gemm_plan_trace", "gemm_plan_clock_log", "gemm_plan_destroy", "gemm_probe_mma_rate",
              "gemm_probe_mma_rate_n"):
    getattr(_lib, _name).restype = _int


class GemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {gemm_strerror(status)} ({status})")


def _check(rc: int, where: str) -> int:
    if rc != GEMM_OK:
        raise GemmError(rc, where)
    return rc


def gemm_strerror(status: int) -> str:
    return _lib.gemm_strerror(int(status)).decode()


def gemm_plan_create(device: int = -1, flags: int = 0) -> int:
    h = _vp()
    _check(_lib.gemm_plan_create(ctypes.byref(h), int(device), int(flags)), "gemm_plan_create")
    return h.value


def gemm_plan_set_option(plan: int, option: int, value: int) -> None:
    _check(_lib.gemm_plan_set_option(_vp(plan), int(option), int(value)), "gemm_plan_set_option")


def gemm_run(A: int, B: int, C: int, M: int, N: int, K: int, dtype: int, out_dtype: int,
             stream: int = 0) -> None:
    _check(_lib.gemm_run(_vp(A), _vp(B), _vp(C), M, N, K, dtype, out_dtype, _vp(stream)), "gemm_run")


def gemm_run_noalloc(A: int, B: int, C: int, M: int, N: int, K: int, dtype: int, out_dtype: int,
                     stream: int = 0) -> None:
    """Allocation-free gemm_run: for callers that may not allocate device memory
    (services whose pool owns all of HBM, embedders under a foreign allocator,
    loops that cannot take a cudaFree's device-wide synchronisation).  The
    first call on a device sets that device up; make it before any stream
    capture.  Calls that overlap on the GPU share one status record and race."""
    _check(_lib.gemm_run_noalloc(_vp(A), _vp(B), _vp(C), M, N, K, dtype, out_dtype, _vp(stream)),
           "gemm_run_noalloc")


def gemm_probe_mma_rate(dtype: int = 0, cta_pair: int = 2, mmas_per_sm: int = 1 << 16, tile_n: int = 256) -> dict:
    """Tensor-core issue-rate probe on the current device (see include/gemm.h):
    back-to-back MMAs of the GEMM's shape (N = tile_n) on every SM, no loads."""
    fpc, tf, mhz = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    _check(_lib.gemm_probe_mma_rate_n(int(dtype), int(cta_pair), int(tile_n), int(mmas_per_sm), ctypes.byref(fpc),
                                      ctypes.byref(tf), ctypes.byref(mhz)), "gemm_probe_mma_rate_n")
    return {"flop_per_clk_per_sm": fpc.value, "tflops": tf.value, "sm_mhz": mhz.value}


def gemm_plan_run(plan: int, A: int, B: int, C: int, M: int, N: int, K: int, dtype: int,
                  out_dtype: int, stream: int = 0) -> None:
    _check(_lib.gemm_plan_run(_vp(plan), _vp(A), _vp(B), _vp(C), M, N, K, dtype, out_dtype,
                              _vp(stream)), "gemm_plan_run")


def gemm_plan_run_layout(plan: int, A: int, B: int, C: int, M: int, N: int, K: int, dtype: int,
                         out_dtype: int, layout: int, stream: int = 0) -> None:
    _check(_lib.gemm_plan_run_layout(_vp(plan), _vp(A), _vp(B), _vp(C), M, N, K, dtype, out_dtype, layout,
                                     _vp(stream)), "gemm_plan_run_layout")


def gemm_plan_run_batched(plan: int, A: int, B: int, C: int, batch: int, M: int, N: int, K: int, stride_a: int,
                          stride_b: int, stride_c: int, dtype: int, out_dtype: int, layout: int = 0,
                          stream: int = 0) -> None:
    _check(_lib.gemm_plan_run_batched(_vp(plan), _vp(A), _vp(B), _vp(C), batch, M, N, K, stride_a, stride_b,
                                      stride_c, dtype, out_dtype, layout, _vp(stream)), "gemm_plan_run_batched")


def gemm_plan_run_host(plan: int, A_host: int, B_host: int, C_host: int, M: int, N: int, K: int,
                       dtype: int, out_dtype: int, stream: int = 0) -> None:
    _check(_lib.gemm_plan_run_host(_vp(plan), _vp(A_host), _vp(B_host), _vp(C_host), M, N, K,
                                   dtype, out_dtype, _vp(stream)), "gemm_plan_run_host")


def gemm_plan_status(plan: int) -> int:
    st = _int(0)
    _check(_lib.gemm_plan_status(_vp(plan), ctypes.byref(st)), "gemm_plan_status")
    return st.value


def gemm_plan_last_grid(plan: int) -> int:
    n = _int(0)
    _check(_lib.gemm_plan_last_grid(_vp(plan), ctypes.byref(n)), "gemm_plan_last_grid")
    return n.value


def gemm_plan_last_split(plan: int) -> int:
    v = _int()
    _check(_lib.gemm_plan_last_split(_vp(plan), ctypes.byref(v)), "gemm_plan_last_split")
    return v.value


def gemm_plan_last_tile_n(plan: int) -> int:
    n = _int(0)
    _check(_lib.gemm_plan_last_tile_n(_vp(plan), ctypes.byref(n)), "gemm_plan_last_tile_n")
    return n.value


def gemm_plan_last_launch(plan: int) -> dict:
    v = [_int(0) for _ in range(5)]
    _check(_lib.gemm_plan_last_launch(_vp(plan), *[ctypes.byref(x) for x in v]), "gemm_plan_last_launch")
    keys = ("ctas", "ctas_per_unit", "tile_n", "dp_waves", "sk_tiles")
    return {k: x.value for k, x in zip(keys, v)}


def gemm_plan_trace(plan: int):
    """Timeline words of a GEMM_TRACE build as a [ctas, slots] uint64 array."""
    import numpy as np
    ctas, slots = _int(0), _int(0)
    _lib.gemm_plan_trace(_vp(plan), None, 0, ctas, slots)
    buf = np.zeros((ctas.value, slots.value), dtype=np.uint64)
    _check(_lib.gemm_plan_trace(_vp(plan), buf.ctypes.data_as(_vp), buf.nbytes, ctypes.byref(ctas),
                                ctypes.byref(slots)), "gemm_plan_trace")
    return buf


def gemm_plan_clock_log(plan: int, capacity: int = 1 << 16) -> list:
    """(SM cycles, ns) of CTA 0's lifetime for each launch since the last
    read, oldest first (GEMM_OPT_CLOCK_LOG must be set); empties the log."""
    buf = (ctypes.c_uint64 * (2 * capacity))()
    n = _i64(0)
    _check(_lib.gemm_plan_clock_log(_vp(plan), buf, capacity, ctypes.byref(n)), "gemm_plan_clock_log")
    return [(int(buf[2 * i]), int(buf[2 * i + 1])) for i in range(n.value)]


def gemm_plan_destroy(plan: int) -> None:
    _check(_lib.gemm_plan_destroy(_vp(plan)), "gemm_plan_destroy")


def raw_status(fn_name: str, *args) -> int:
    """Call a C entry point with raw ctypes arguments and return its status code
    (used by tests that check error returns)."""
    return int(getattr(_lib, fn_name)(*args))


# ------------------------------------------------------------------ torch helpers

def _dtype_code(t) -> int:
    import torch
    codes = {torch.bfloat16: GEMM_BF16, torch.float16: GEMM_F16, torch.float32: GEMM_F32,
             torch.float8_e4m3fn: GEMM_E4M3, torch.float8_e5m2: GEMM_E5M2}
    if t not in codes:
        raise TypeError(f"unsupported dtype {t}")
    return codes[t]


_default_plans = {}


def _check_devices(A, B):
    """The library reads and writes device memory only: both operands must be
    CUDA tensors on one device (a host pointer handed to the kernel would be
    read as a device address)."""
    if not (getattr(A, "is_cuda", False) and getattr(B, "is_cuda", False)):
        raise ValueError("A and B must be CUDA tensors (gemm_plan_run_host takes host buffers)")
    if A.device != B.device:
        raise ValueError("A and B must be on the same device")


def default_plan(device=None) -> int:
    """A plan for `device` (torch device or index; default: the current one),
    created on first use and kept for the life of the process; what
    matmul() and bmm() use when no plan is passed."""
    import torch
    if device is None:
        idx = torch.cuda.current_device()
    else:
        d = torch.device("cuda", device) if isinstance(device, int) else torch.device(device)
        idx = d.index if d.index is not None else torch.cuda.current_device()
    if idx not in _default_plans:
        _default_plans[idx] = gemm_plan_create(idx)
    return _default_plans[idx]


def matmul(A, B, out_dtype=None, plan: Optional[int] = None, out=None, a_km: bool = False,
           b_kn: bool = False):
    """C = A @ B.T for CUDA tensors A [M,K], B [N,K] (contiguous; bf16, f16,
    float8_e4m3fn or float8_e5m2, both the same).

    a_km / b_kn: A is given as [K,M] / B as [K,N] (both contiguous), read in
    place by the tensor cores (16-bit inputs), so ``matmul(A, B, b_kn=True)``
    is the plain A @ B.
    out_dtype: torch.float32, torch.bfloat16 or torch.float16 (default: A's
    dtype for 16-bit inputs, bf16 for fp8 inputs).
    plan: default_plan(A.device) when omitted.
    Runs on torch's current stream of A's device.
    """
    import torch
    _check_devices(A, B)
    if A.dim() != 2 or B.dim() != 2:
        raise ValueError("A and B must be matrices")
    layout = (GEMM_A_MN_MAJOR if a_km else 0) | (GEMM_B_MN_MAJOR if b_kn else 0)
    if a_km:
        A = A.t()          # view only: the data stay K-by-M
    if b_kn:
        B = B.t()
    if A.shape[1] != B.shape[1]:
        raise ValueError("the operands' K extents differ")
    if A.dtype != B.dtype:
        raise TypeError("A and B must have the same dtype")
    if not ((A.t() if a_km else A).is_contiguous() and (B.t() if b_kn else B).is_contiguous()):
        raise ValueError("A and B must be contiguous row-major")
    if out_dtype is None:
        out_dtype = A.dtype if A.element_size() == 2 else torch.bfloat16
    M, K = A.shape
    N = B.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=A.device)
    elif out.shape != (M, N) or out.dtype != out_dtype or not out.is_contiguous() or out.device != A.device:
        raise ValueError("out must be a contiguous [M,N] tensor of out_dtype on A's device")
    stream = torch.cuda.current_stream(A.device).cuda_stream
    if plan is None:
        plan = default_plan(A.device)
    args = (A.data_ptr(), B.data_ptr(), out.data_ptr(), M, N, K, _dtype_code(A.dtype),
            _dtype_code(out_dtype), stream)
    with torch.cuda.device(A.device):   # the library runs on the current device: the operands'
        if layout:
            gemm_plan_run_layout(plan, *args[:-1], layout, args[-1])
        else:
            gemm_plan_run(plan, *args)
    return out


def bmm(A, B, plan: Optional[int] = None, out_dtype=None, out=None):
    """C[e] = A[e] @ B[e].T for CUDA tensors A [batch,M,K] or [M,K] (shared) and
    B [batch,N,K] or [N,K] (shared), contiguous, same 16-bit or 8-bit dtype,
    in one launch (gemm_plan_run_batched; plan: default_plan(A.device) when
    omitted).  Returns C [batch,M,N]."""
    import torch
    _check_devices(A, B)
    if A.dim() not in (2, 3) or B.dim() not in (2, 3) or A.shape[-1] != B.shape[-1]:
        raise ValueError("A must be [batch,M,K] or [M,K], B [batch,N,K] or [N,K]")
    if A.dtype != B.dtype or not (A.is_contiguous() and B.is_contiguous()):
        raise ValueError("A and B must be contiguous and of one dtype")
    batch = A.shape[0] if A.dim() == 3 else B.shape[0] if B.dim() == 3 else 1
    if (A.dim() == 3 and A.shape[0] != batch) or (B.dim() == 3 and B.shape[0] != batch):
        raise ValueError("batch extents differ")
    M, K = A.shape[-2], A.shape[-1]
    N = B.shape[-2]
    if out_dtype is None:
        out_dtype = A.dtype if A.element_size() == 2 else torch.bfloat16
    if out is None:
        out = torch.empty((batch, M, N), dtype=out_dtype, device=A.device)
    elif out.shape != (batch, M, N) or out.dtype != out_dtype or not out.is_contiguous() or out.device != A.device:
        raise ValueError("out must be a contiguous [batch,M,N] tensor of out_dtype on A's device")
    if plan is None:
        plan = default_plan(A.device)
    sa = M * K if A.dim() == 3 else 0
    sb = N * K if B.dim() == 3 else 0
    with torch.cuda.device(A.device):
        gemm_plan_run_batched(plan, A.data_ptr(), B.data_ptr(), out.data_ptr(), batch, M, N, K, sa, sb, M * N,
                              _dtype_code(A.dtype), _dtype_code(out_dtype), 0,
                              torch.cuda.current_stream(A.device).cuda_stream)
    return out
