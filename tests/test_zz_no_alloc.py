"""gemm_nt_f16_f32_batched_no_alloc: the batched product with no device
allocation, for callers that must not allocate (code being captured into a
CUDA graph cannot call cudaMalloc; an application whose pool allocator owns the
device memory may not allow a library to take more; a latency-critical first
call cannot pay for one).  The entry point keeps its scratch in one fixed
array inside the library, which keeps the previous call's contents.  So on
two calls in a row its answers must
  * lie within the parity tolerance of the CPU oracle (bit for bit with
    integer-valued inputs, whose every partial sum is exact in fp32), and
  * equal, bit for bit, the ordinary entry point's answer: both run the same
    kernel with the same plan, and the split's partial sums are added in a
    fixed k order;
and a split too large for that array must be refused, not attempted.

Collected last on purpose (file name), so a failure here stops a -x run only
after every other test has run.  It needs nothing from earlier tests and also
passes alone in a fresh process.
"""
import numpy as np
import pytest

import dense_fp16_tensor_gemm_gb300 as gnt
import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from dense_fp16_tensor_gemm_gb300 import _build
    _build.build()
    return gnt.load()


def _call(fn, a, b, out, batch, M, N, K):
    import torch
    return fn(a.data_ptr(), b.data_ptr(), out.data_ptr(), M, N, K, K, K, N, M * K, N * K, M * N, batch,
              torch.cuda.current_stream().cuda_stream)


def _run(lib, fn, a, b, batch, M, N, K):
    import torch
    out = torch.full((batch, M, N), float("nan"), dtype=torch.float32, device="cuda")
    assert _call(fn, a, b, out, batch, M, N, K) == 0
    gnt.gemm_nt_check()
    return out.cpu().numpy()


@pytest.mark.parametrize("batch,M,N,K,dist", [
    (1, 512, 512, 8192, "normal"),   # 4 tiles, long K: split across pairs, scratch in use
    (1, 300, 500, 6144, "normal"),   # ragged, 4 tiles, split
    (1, 512, 512, 8192, "int4"),     # split, integer-valued: exact
    (2, 300, 500, 640, "normal"),    # short K: whole tiles, no scratch needed
])
def test_matches_oracle_and_existing_entry_point_on_consecutive_calls(lib, batch, M, N, K, dist):
    import torch
    A, B = workloads.make_inputs(batch, M, N, K, dist, 1.0, seed=M + N + K)
    ref, absdot = oracle.gemm_nt(A, B)
    a, b = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    existing = _run(lib, lib.gemm_nt_f16_f32_batched, a, b, batch, M, N, K)
    for call in range(2):  # the array keeps the previous call's contents
        got = _run(lib, lib.gemm_nt_f16_f32_batched_no_alloc, a, b, batch, M, N, K)
        assert not np.isnan(got).any(), "call %d left elements unwritten" % call
        if dist == "int4":
            bad = got.astype(np.float64) != ref
            assert not bad.any(), "call %d: %d elements differ from the exact result" % (call, int(bad.sum()))
        else:
            ok = oracle.within_tolerance(got, ref, absdot)
            assert ok.all(), "call %d: %d elements outside the oracle's tolerance" % (call, int((~ok).sum()))
        assert np.array_equal(got, existing), \
            "call %d: %d elements differ from the existing entry point" % (call, int((got != existing).sum()))


def test_split_beyond_the_array_is_refused(lib):
    """16 tiles with K = 8192 would split over 64 CTA pairs, more than the 16
    the fixed array holds: the call returns SCRATCH_TOO_SMALL and writes nothing."""
    import torch
    M = N = 1024
    K = 8192
    a = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    b = torch.zeros((N, K), dtype=torch.float16, device="cuda")
    out = torch.full((1, M, N), 7.0, dtype=torch.float32, device="cuda")
    assert _call(lib.gemm_nt_f16_f32_batched_no_alloc, a, b, out, 1, M, N, K) == gnt.Status.SCRATCH_TOO_SMALL
    gnt.gemm_nt_check()
    assert bool(torch.all(out == 7.0))
    assert "scratch" in gnt.error_string(gnt.Status.SCRATCH_TOO_SMALL)
