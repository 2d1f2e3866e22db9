"""The CPU oracle against its pins, and planted mistakes that the pins catch.

No GPU.  Each planted mistake is a textual change to a private copy of
oracle/gemm_oracle.c (the oracle itself is never modified): a dropped term, a
transposed operand, wrong signs, an off-by-one exponent bias, a broken
subnormal scale, ties rounded away from even, a wrong row stride, a missing
absolute value, a wrong sampled index, and in the 8-bit decoder a
wrong special-value rule, bias, field widths, subnormal scale or format.  Every one must fail at least one pin.
"""
import os
import shutil

import numpy as np
import pytest

import oracle
from tests import oracle_pins


@pytest.fixture(scope="module")
def real_oracle():
    return oracle.default()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(real_oracle, pin):
    pin(real_oracle)


# (description, text in gemm_oracle.c, replacement)
MUTANTS = [
    ("drops the last k term", "for (int64_t k = 0; k < K; ++k) {\n                const double p = ai[k] * bj[k];",
     "for (int64_t k = 0; k + 1 < K; ++k) {\n                const double p = ai[k] * bj[k];"),
    ("reads B as K×N instead of N×K", "const double p = ai[k] * bj[k];",
     "const double p = ai[k] * b[k * N + j];"),
    ("negates the first product", "                acc += p;\n                mag += fabs(p);\n            }\n            C[i * N + j]",
     "                acc += (k == 0 ? -p : p);\n                mag += fabs(p);\n            }\n            C[i * N + j]"),
    ("exponent bias off by one", "const int bias = (1 << (eb - 1)) - 1;\n    const int sign",
     "const int bias = (1 << (eb - 1));\n    const int sign"),
    ("subnormal scale off by one", "v = ldexp((double)f, 1 - bias - fb);",
     "v = ldexp((double)f, -bias - fb);"),
    ("rounds ties away from zero", "if (rem > 0.5 || (rem == 0.5 && (n & 1))) n += 1;",
     "if (rem >= 0.5) n += 1;"),
    ("wrong row stride of A", "const double* ai = a + i * K;", "const double* ai = a + i;"),
    ("magnitude sum without abs", "                mag += fabs(p);\n            }\n            C[i * N + j]",
     "                mag += p;\n            }\n            C[i * N + j]"),
    ("sampled entries swap row and column", "const int64_t ra = I[t] * K, rb = J[t] * K;",
     "const int64_t ra = (J[t] < M ? J[t] : I[t]) * K, rb = (I[t] < N ? I[t] : J[t]) * K;"),
    ("E4M3 all-ones exponent read as infinity", "if (dtype == ORACLE_E4M3 && e == 15 && f == 7) {\n        v = NAN;",
     "if (dtype == ORACLE_E4M3 && e == 15) {\n        v = (f == 0) ? INFINITY : NAN;"),
    ("fp8 exponent bias off by one", "const int bias8 = (1 << (eb - 1)) - 1;", "const int bias8 = (1 << (eb - 1));"),
    ("E5M2 read with E4M3 field widths", "const int eb = dtype == ORACLE_E4M3 ? 4 : 5, fb = dtype == ORACLE_E4M3 ? 3 : 2;",
     "const int eb = 4, fb = 3;"),
    ("fp8 subnormal scale off by one", "v = ldexp((double)f, 1 - bias8 - fb);", "v = ldexp((double)f, -bias8 - fb);"),
    ("fp8 bytes decoded as f16 patterns", "return oracle_decode8(((const uint8_t*)bits)[idx], dtype);",
     "return oracle_decode16((uint16_t)((const uint8_t*)bits)[idx], ORACLE_F16);"),
    ("overflow saturates instead of going to infinity",
     "if (e_field >= emax_field) return sign | (uint16_t)((uint32_t)emax_field << fb);  /* overflow */",
     "if (e_field >= emax_field) return sign | (uint16_t)(((uint32_t)(emax_field - 1) << fb) | ((1u << fb) - 1));"),
]


@pytest.mark.parametrize("desc,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, desc, old, new):
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation anchor not unique/found: {desc}"
    mutated = tmp_path / "gemm_oracle_mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.build(force=True, src=str(mutated), out=str(tmp_path / "libmutant.so"))
    mutant = oracle.Oracle(lib)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mutant)
        except AssertionError:
            failed.append(pin.__name__)
        except Exception as e:  # a crash in a mutant also counts as caught
            failed.append(f"{pin.__name__}:{type(e).__name__}")
    assert failed, f"no pin caught the planted mistake: {desc}"


@pytest.mark.parametrize("name,shape", [("gemm_256_f32out", None), ("gemm_ragged_4000x3000x5000", (1000, 760, 1256)),
                                        ("gemm_1024x4096x4096_f16", (264, 392, 1024))])
def test_torch_fp32_second_opinion(real_oracle, name, shape):
    """An untrusted second opinion: torch's CPU matmul in fp32 on the inputs
    widened exactly to fp32 agrees with the oracle within the fp32
    accumulation bound |C - C_ref| <= 1e-5 * S used for the kernel (the
    256³ workload, and the ragged and f16 workloads' distributions at sizes
    that still span several tiles)."""
    import torch
    import workloads as wl
    w = wl.WORKLOADS[name]
    A, B = wl.make_inputs(w) if shape is None else wl.make_inputs(w, *shape, seed=w.seed + 100)
    C_ref, S = real_oracle.gemm(wl.as_bits(A), wl.as_bits(B), w.dtype)
    C_t = torch.matmul(A.float(), B.float().t()).double().numpy()
    assert np.all(np.abs(C_t - C_ref) <= 1e-5 * S), float(np.max(np.abs(C_t - C_ref) / S))
