"""The C-ABI library without a GPU: it builds, loads, exports every symbol
include/*.h declares, and rejects bad arguments on the host before any CUDA
call.  No compute calls are made here."""
import ctypes
import glob
import os
import re

import pytest

import __graft_entry__ as entry

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M):
            if m.group(1) not in ("if", "while", "for", "return", "sizeof"):
                names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    entry.build()
    import dense_gemm_blackwell_persistent_gb300 as g
    return g


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("gemm_plan_create", "gemm_run", "gemm_plan_destroy", "gemm_plan_run", "gemm_strerror",
                     "gemm_plan_run_layout"):
        assert required in names, names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(lib.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), f"{name} declared in include/ but not exported"


def test_host_validation_without_gpu(lib):
    vp = ctypes.c_void_p
    rs = lib.raw_status
    good = vp(1 << 20)
    # bad dtype pair
    assert rs("gemm_run", good, good, good, 64, 64, 64, 2, 2, None) == lib.GEMM_ERR_INVALID_ARG
    assert rs("gemm_run", good, good, good, 64, 64, 64, 0, 7, None) == lib.GEMM_ERR_INVALID_ARG
    assert rs("gemm_run", good, good, good, 64, 64, 64, 5, 2, None) == lib.GEMM_ERR_INVALID_ARG
    assert rs("gemm_run", good, good, good, 64, 64, 64, 0, 3, None) == lib.GEMM_ERR_INVALID_ARG   # fp8 out
    # negative sizes
    assert rs("gemm_run", good, good, good, -1, 64, 64, 0, 2, None) == lib.GEMM_ERR_INVALID_ARG
    # null pointers
    assert rs("gemm_run", None, good, good, 64, 64, 64, 0, 2, None) == lib.GEMM_ERR_INVALID_ARG
    assert rs("gemm_run", good, good, None, 64, 64, 64, 0, 2, None) == lib.GEMM_ERR_INVALID_ARG
    # misaligned pointers
    assert rs("gemm_run", vp((1 << 20) + 8), good, good, 64, 64, 64, 0, 2, None) == lib.GEMM_ERR_MISALIGNED
    assert rs("gemm_run", good, good, vp((1 << 20) + 4), 64, 64, 64, 0, 2, None) == lib.GEMM_ERR_MISALIGNED
    # pitches TMA cannot address (K bytes and N bytes multiples of 16)
    assert rs("gemm_run", good, good, good, 64, 64, 60, 0, 2, None) == lib.GEMM_ERR_UNSUPPORTED
    assert rs("gemm_run", good, good, good, 64, 64, 24, 3, 2, None) == lib.GEMM_ERR_UNSUPPORTED   # fp8: K % 16
    assert rs("gemm_run", good, good, good, 64, 64, 24, 4, 2, None) == lib.GEMM_ERR_UNSUPPORTED
    assert rs("gemm_run", good, good, good, 64, 6, 64, 0, 0, None) == lib.GEMM_ERR_UNSUPPORTED
    assert rs("gemm_run", good, good, good, 64, 2, 64, 0, 2, None) == lib.GEMM_ERR_UNSUPPORTED
    assert rs("gemm_run", good, good, good, 1 << 31, 64, 64, 0, 2, None) == lib.GEMM_ERR_UNSUPPORTED
    for big in ((1 << 31) - 1016, 1 << 40):   # beyond the largest extent (2^31 - 1024) in M, N or K
        assert rs("gemm_run", good, good, good, big, 64, 64, 0, 2, None) == lib.GEMM_ERR_UNSUPPORTED
        assert rs("gemm_run", good, good, good, 64, big, 64, 0, 2, None) == lib.GEMM_ERR_UNSUPPORTED
        assert rs("gemm_run", good, good, good, 64, 64, big, 0, 2, None) == lib.GEMM_ERR_UNSUPPORTED
    # empty problems are a no-op and touch nothing
    assert rs("gemm_run", None, None, None, 0, 64, 64, 0, 2, None) == lib.GEMM_OK
    assert rs("gemm_run", None, None, None, 64, 0, 64, 0, 2, None) == lib.GEMM_OK
    # null plan handles
    assert rs("gemm_plan_run", None, good, good, good, 64, 64, 64, 0, 2, None) == lib.GEMM_ERR_INVALID_ARG
    assert rs("gemm_plan_destroy", None) == lib.GEMM_ERR_INVALID_ARG
    assert rs("gemm_plan_set_option", None, 1, ctypes.c_int64(2)) == lib.GEMM_ERR_INVALID_ARG
    assert rs("gemm_plan_create", None, -1, 0) == lib.GEMM_ERR_INVALID_ARG
    # the tensor-core probe checks its arguments before touching the device
    assert rs("gemm_probe_mma_rate", 2, 2, 1 << 12, None, None, None) == lib.GEMM_ERR_INVALID_ARG   # fp32 operands
    assert rs("gemm_probe_mma_rate", 0, 4, 1 << 12, None, None, None) == lib.GEMM_ERR_INVALID_ARG   # 4 CTAs
    assert rs("gemm_probe_mma_rate", 0, 2, 6, None, None, None) == lib.GEMM_ERR_INVALID_ARG         # not whole k-blocks
    for n in (0, 8, 100, 272):                                                                      # not an MMA width
        assert rs("gemm_probe_mma_rate_n", 0, 2, n, 1 << 12, None, None, None) == lib.GEMM_ERR_INVALID_ARG
    # the clock log checks its arguments before touching the device
    n = ctypes.c_int64(0)
    assert rs("gemm_plan_clock_log", None, None, 0, ctypes.byref(n)) == lib.GEMM_ERR_INVALID_ARG
    for code in range(-9, 1):
        assert lib.gemm_strerror(code) != "unknown status"


def test_no_device_is_reported(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(lib.GemmError) as e:
        lib.gemm_plan_create(-1)
    assert e.value.status == lib.GEMM_ERR_NO_DEVICE
    vp = ctypes.c_void_p
    good = vp(1 << 20)
    # a well-formed call with no device: fails cleanly, enqueues nothing
    assert lib.raw_status("gemm_run", good, good, good, 64, 64, 64, 0, 2, None) == lib.GEMM_ERR_NO_DEVICE
    assert lib.raw_status("gemm_probe_mma_rate", 0, 2, 1 << 12, None, None, None) == lib.GEMM_ERR_NO_DEVICE


def test_product_path_has_no_cpu_fallback():
    """The package never imports the oracle and has no Python arithmetic path."""
    pkg = os.path.join(ROOT, "dense_gemm_blackwell_persistent_gb300")
    for path in glob.glob(os.path.join(pkg, "**", "*.py"), recursive=True) + \
            glob.glob(os.path.join(pkg, "csrc", "*")):
        text = open(path).read()
        assert "oracle" not in text.replace("oracle/", ""), path
        for forbidden in ("torch.matmul", "np.matmul", "np.dot", "einsum", "torch.mm("):
            assert forbidden not in text, (path, forbidden)


def test_torch_helpers_refuse_host_tensors(lib):
    """matmul() and bmm() hand device pointers to the library: host tensors are
    refused before anything reaches it (they would be read as device
    addresses); host buffers go through gemm_plan_run_host instead."""
    import torch
    A = torch.zeros((64, 64), dtype=torch.bfloat16)
    B = torch.zeros((32, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensors"):
        lib.matmul(A, B)
    with pytest.raises(ValueError, match="CUDA tensors"):
        lib.matmul(A, B.t().contiguous(), b_kn=True)
    with pytest.raises(ValueError, match="CUDA tensors"):
        lib.bmm(A.view(1, 64, 64), B)


def build_c_caller(lib_path, exe):
    """Compile tests/native/c_caller.c as strict C99 against include/gemm.h and
    link it to the library (rpath to the library's folder)."""
    import subprocess
    src = os.path.join(ROOT, "tests", "native", "c_caller.c")
    lib_dir = os.path.dirname(lib_path)
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-O1", "-I", os.path.join(ROOT, "include"),
           src, "-o", exe, "-L", lib_dir, "-l:" + os.path.basename(lib_path), "-Wl,-rpath," + lib_dir]
    subprocess.run(cmd, check=True, capture_output=True, text=True)


def test_plain_c_caller_compiles_and_links(lib, tmp_path):
    """The header is valid C99 without CUDA headers, and a C program that
    calls the boundary links against the library (run on a GPU by the GPU
    tests; here only with --link-only, which exits before any call)."""
    import subprocess
    exe = str(tmp_path / "c_caller")
    build_c_caller(lib.LIB_PATH, exe)
    assert subprocess.run([exe, "--link-only"]).returncode == 0
