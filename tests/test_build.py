"""Build properties of the kernel, checked without a GPU: ptxas's own report
(-Xptxas -v: target, registers, stack, spills) for representative
instantiations.  The report names the target each entry function was
assembled for, which must be sm_103a.

The persistent kernel keeps one CTA per SM with 192 threads, so registers
are not what limits residency, but a spill would put local-memory traffic
inside the K loop and the epilogue.  Every instantiation compiled here must
report zero stack frame and zero spill bytes."""
import os
import re
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "dense_gemm_blackwell_persistent_gb300", "csrc")
INCLUDE = os.path.join(ROOT, "include")

# (CTAs per unit, output type, operand width, padded MN-major B, extra defines): pairs with bf16
# C (the benchmark's kernel), the 4-CTA multicast unit with fp32 C, 8-bit operands, the padded
# form, and the benchmark's kernel in the GEMM_DEBUG build (its checks must not spill either)
CASES = [(2, 0, 0, 0, ""), (4, 2, 0, 0, ""), (2, 0, 1, 0, ""), (1, 1, 0, 1, ""), (2, 0, 0, 0, "-DGEMM_DEBUG")]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return None


def _ptxas_report(case, tmp):
    cluster, out, inp, pad, extra = case
    cmd = [_nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "--expt-relaxed-constexpr",
           "-Xptxas", "-v", "-I", INCLUDE, "-I", CSRC, f"-DGEMM_INST_CLUSTER={cluster}", f"-DGEMM_INST_OUT={out}",
           f"-DGEMM_INST_IN={inp}", f"-DGEMM_INST_BMN={pad}", *([extra] if extra else []), "-c",
           os.path.join(CSRC, "kernels_inst.cu"),
           "-o", os.path.join(tmp, "k_{}_{}_{}_{}{}.o".format(*case[:4], "_dbg" if extra else ""))]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr[-2000:]
    return res.stdout + res.stderr


def test_no_spills_in_the_kernel(tmp_path):
    if _nvcc() is None:
        pytest.skip("nvcc not found")
    with ThreadPoolExecutor(len(CASES)) as ex:
        reports = list(ex.map(lambda c: _ptxas_report(c, str(tmp_path)), CASES))
    for case, rep in zip(CASES, reports):
        entries = re.findall(r"Compiling entry function '(\w+)' for '(sm_\w+)'", rep)
        assert entries and all(arch == "sm_103a" for _, arch in entries), (case, entries)
        entries = [name for name, _ in entries]
        frames = re.findall(r"(\d+) bytes stack frame, (\d+) bytes spill stores, (\d+) bytes spill loads", rep)
        regs = [int(r) for r in re.findall(r"Used (\d+) registers", rep)]
        assert entries and len(frames) == len(entries) == len(regs), (case, rep[-2000:])
        for name, (stack, st, ld), r in zip(entries, frames, regs):
            assert (int(stack), int(st), int(ld)) == (0, 0, 0), (case, name, stack, st, ld)
            assert r <= 255, (case, name, r)
