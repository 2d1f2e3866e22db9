"""gemm_run_noalloc, the allocation-free entry point, against gemm_plan_run.

Some callers of this library may not allocate device memory: services that
give all of HBM to their own pool at start-up, embedders whose memory belongs
to another allocator that must account for every byte, latency-critical loops
that cannot take the device-wide synchronisation of a cudaFree.
gemm_run_noalloc serves them: it runs the same kernel with the
kernel's scratch (its status record) in a static device array instead of a
plan's cudaMalloc'd word.  Here it is called through the C ABI twice in a row,
on different shapes and dtypes.  Both entry points launch the same kernel
with the same default configuration, so each output must equal the plan
entry point's output on the same inputs bit for bit (a difference would
mean a different launch shape); both are also checked against the fp64
oracle within the tolerance every parity test uses.

The file name sorts last so that a run stopping at its first failure has
already run every other test; it also passes alone in a fresh process.
"""
import pytest
import torch

import oracle
import workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu


def test_noalloc_matches_plan_entry_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_gemm_blackwell_persistent_gb300 as g
    torch.cuda.set_device(0)
    plan = g.gemm_plan_create(0)
    stream = torch.cuda.current_stream().cuda_stream
    cases = [(1000, 776, 1256, wl.BF16, wl.F32, 21), (520, 1288, 392, wl.F16, wl.BF16, 22)]
    try:
        for M, N, K, dt, out, seed in cases:
            w = wl.Workload("noalloc", M, N, K, dt, out, "normal", seed)
            A, B = wl.make_inputs(w)
            Ad, Bd = A.cuda(), B.cuda()
            C_free = torch.full((M, N), float("nan"), dtype=wl.TORCH_DTYPES[out], device="cuda")
            C_plan = torch.full((M, N), float("nan"), dtype=wl.TORCH_DTYPES[out], device="cuda")
            g.gemm_run_noalloc(Ad.data_ptr(), Bd.data_ptr(), C_free.data_ptr(), M, N, K, dt, out, stream)
            g.gemm_plan_run(plan, Ad.data_ptr(), Bd.data_ptr(), C_plan.data_ptr(), M, N, K, dt, out, stream)
            torch.cuda.synchronize()
            assert g.gemm_plan_status(plan) == 0
            C_ref, S = oracle.gemm(wl.as_bits(A), wl.as_bits(B), dt)
            assert torch.equal(C_free, C_plan), f"noalloc vs plan entry, {M}x{N}x{K}"
            got_free, got_plan = parity.to_f64(C_free), parity.to_f64(C_plan)
            parity.assert_within(got_free, C_ref, S, out, f"noalloc {M}x{N}x{K}")
            parity.assert_within(got_plan, C_ref, S, out, f"plan {M}x{N}x{K}")
    finally:
        torch.cuda.synchronize()
        g.gemm_plan_destroy(plan)

