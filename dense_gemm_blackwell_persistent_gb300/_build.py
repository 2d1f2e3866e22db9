"""Build the CUDA library in-tree with nvcc (sm_103a only).

Produces ``dense_gemm_blackwell_persistent_gb300/_lib/libgb300gemm.so`` from
``csrc/gemm_api.cu`` (host side), ``csrc/mma_probe.cu`` (the tensor-core
issue-rate probe) and 24 objects of ``csrc/kernels_inst.cu``
(one per unit size × output type × operand width, plus the padded MN-major-B
forms), compiled in parallel.  The CUDA
runtime is linked statically and the driver's tensor-map encoder is looked up
at run time, so the library loads on a machine without a GPU.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libgb300gemm.so")
# Build variants: "" is the product library; "trace" adds -DGEMM_TRACE
# (per-CTA timeline stamps, read back with gemm_plan_trace); "debug" adds
# -DGEMM_DEBUG (consistency checks of tile coordinates, ring stage and phase,
# k-block ranges and store boxes inside the kernel, reported as
# GEMM_ERR_INTERNAL through gemm_plan_status).
VARIANT_DEFINES = {"": [], "trace": ["-DGEMM_TRACE"], "debug": ["-DGEMM_DEBUG"]}


def lib_path(variant: str = "") -> str:
    if variant not in VARIANT_DEFINES:
        raise ValueError(f"unknown library variant {variant!r}")
    return LIB if not variant else os.path.join(LIBDIR, f"libgb300gemm_{variant}.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC",
    "--expt-relaxed-constexpr",
]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + glob.glob(os.path.join(INCLUDE, "*.h")))


def up_to_date(variant: str = "") -> bool:
    lib = lib_path(variant)
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(s) <= t for s in _sources())


# (CTAs per unit, output type, operand width) variants of the kernel, one
# object file each
VARIANTS = [(cluster, out, inp, 0) for cluster in (1, 2, 4) for out in (0, 1, 2) for inp in (0, 1)]
VARIANTS += [(cluster, out, 0, 1) for cluster in (1, 2) for out in (0, 1, 2)]   # padded MN-major B


def _compile(args):
    cmd, verbose = args
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed ({res.returncode}): {' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
    return res.stdout + res.stderr if verbose else ""


def build(force: bool = False, verbose: bool = False, variant: str = "") -> str:
    """Compile every translation unit in parallel, then link the shared library."""
    from concurrent.futures import ThreadPoolExecutor

    lib = lib_path(variant)
    if not force and up_to_date(variant):
        return lib
    os.makedirs(LIBDIR, exist_ok=True)
    objdir = os.path.join(LIBDIR, f"obj{variant}{os.getpid()}")
    os.makedirs(objdir, exist_ok=True)
    nvcc = _nvcc()
    common = [nvcc, *NVCC_FLAGS, *VARIANT_DEFINES[variant], "-I", INCLUDE, "-I", CSRC, "-c"]
    if verbose:
        common.insert(1, "-Xptxas=-v")
    jobs = [(common + [os.path.join(CSRC, "gemm_api.cu"), "-o", os.path.join(objdir, "gemm_api.o")], verbose),
            (common + [os.path.join(CSRC, "mma_probe.cu"), "-o", os.path.join(objdir, "mma_probe.o")], verbose)]
    for cluster, out, inp, pad in VARIANTS:
        obj = os.path.join(objdir, f"kernels_c{cluster}_o{out}_i{inp}_p{pad}.o")
        jobs.append((common + [f"-DGEMM_INST_CLUSTER={cluster}", f"-DGEMM_INST_OUT={out}", f"-DGEMM_INST_IN={inp}",
                               f"-DGEMM_INST_BMN={pad}", os.path.join(CSRC, "kernels_inst.cu"), "-o", obj], verbose))
    workers = max(1, min(len(jobs), os.cpu_count() or 1))
    with ThreadPoolExecutor(workers) as ex:
        logs = list(ex.map(_compile, jobs))
    if verbose:
        print("".join(logs))
    tmp = lib + f".tmp{os.getpid()}"
    objs = sorted(os.path.join(objdir, f) for f in os.listdir(objdir) if f.endswith(".o"))
    link = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-Xcompiler", "-fPIC", *objs, "-o", tmp]
    _compile((link, False))
    os.replace(tmp, lib)
    shutil.rmtree(objdir, ignore_errors=True)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                variant="trace" if "--trace" in sys.argv else "debug" if "--debug" in sys.argv else ""))
