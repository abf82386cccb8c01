"""Failure detection without a GPU fault: every mbarrier wait in the tcgen05
kernels has an iteration limit.  The library's test hooks make one wait run out
on CTA 0 (the producer drops its first stage, or the MMA thread skips its first
stage release); the kernel must give up after the limit, free its TMEM and
return, gemm_nt_check must report GEMM_ERR_DEVICE_TIMEOUT, and the next normal
call on the same context must be correct."""
import numpy as np
import pytest

import dense_fp16_tensor_gemm_gb300 as gnt
import oracle
import workloads
from gpu_util import assert_parity

pytestmark = pytest.mark.gpu

P = gnt.Path
LIMIT = 50_000_000  # SM clock cycles per wait (about 25 ms)


@pytest.fixture(scope="module", autouse=True)
def built():
    from dense_fp16_tensor_gemm_gb300 import _build
    _build.build()
    gnt.load()
    yield
    gnt.gemm_nt_debug_set_fault(0)
    gnt.gemm_nt_debug_set_wait_limit(0)


def _run(A, B, path):
    import torch
    a, b = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    out = torch.zeros((A.shape[0], B.shape[0]), dtype=torch.float32, device="cuda")
    gnt.gemm_nt_f16_f32_batched_path(a.data_ptr(), b.data_ptr(), out.data_ptr(), A.shape[0], B.shape[0],
                                     A.shape[1], A.shape[1], B.shape[1], B.shape[0], 0, 0, 0, 1, path,
                                     torch.cuda.current_stream().cuda_stream)
    return out


@pytest.mark.parametrize("fault", [1, 2])
@pytest.mark.parametrize("path,M,N,K", [(P.TC05, 512, 512, 2048), (P.TC05_PAIR, 512, 512, 2048),
                                        (P.SKINNY, 64, 16384, 2048)])
def test_bounded_wait_reports_timeout(path, M, N, K, fault):
    A, B = workloads.make_inputs(0, M, N, K, "uniform", seed=3)
    gnt.gemm_nt_check()  # clean state
    gnt.gemm_nt_debug_set_wait_limit(LIMIT)
    gnt.gemm_nt_debug_set_fault(fault)
    try:
        _run(A, B, path)
        with pytest.raises(gnt.GemmError) as e:
            gnt.gemm_nt_check()
        assert e.value.status == gnt.Status.DEVICE_TIMEOUT
    finally:
        gnt.gemm_nt_debug_set_fault(0)
        gnt.gemm_nt_debug_set_wait_limit(0)
    # the context is still usable and the status word was cleared
    gnt.gemm_nt_check()
    out = _run(A, B, path)
    gnt.gemm_nt_check()
    ref, absdot = oracle.gemm_nt(A, B)
    assert_parity(out.cpu().numpy(), ref, absdot, what="after timeout " + path.name)


@pytest.mark.parametrize("fault", [1, 2])
@pytest.mark.parametrize("path,M,N,K", [(P.TC05, 256, 384, 2048), (P.TC05_PAIR, 512, 512, 2048),
                                        (P.SKINNY, 64, 16384, 4096)])
def test_bounded_wait_reports_timeout_block_scaled(path, M, N, K, fault):
    """The block-scaled kernels, whose scale copies come from a copier warp
    with waits of its own (on the stage data and the scale ring).  K is long
    enough that every CTA reuses its stages, so a skipped release is waited on."""
    from test_gpu_mx import draw, run_mx
    A, SA, B, SB = draw(1, M, N, K, "e4m3", seed=7)
    gnt.gemm_nt_check()
    gnt.gemm_nt_debug_set_wait_limit(LIMIT)
    gnt.gemm_nt_debug_set_fault(fault)
    try:
        with pytest.raises(gnt.GemmError) as e:
            run_mx(A, SA, B, SB, "e4m3", "f32", path)  # run_mx checks the status
        assert e.value.status == gnt.Status.DEVICE_TIMEOUT
    finally:
        gnt.gemm_nt_debug_set_fault(0)
        gnt.gemm_nt_debug_set_wait_limit(0)
    gnt.gemm_nt_check()
    ref, absdot = oracle.gemm_nt_mx(A, SA, B, SB, dtype="e4m3")
    from gpu_util import check_tol
    check_tol(run_mx(A, SA, B, SB, "e4m3", "f32", path), ref, absdot, "f32", "after timeout mx " + path.name)


@pytest.mark.parametrize("fault", [1, 2])
@pytest.mark.parametrize("path", [P.TC05_M64, P.TC05_WS])
def test_bounded_wait_reports_timeout_other_shapes(path, fault):
    A, B = workloads.make_inputs(0, 64, 1024, 2048, "uniform", seed=5)
    gnt.gemm_nt_check()
    gnt.gemm_nt_debug_set_wait_limit(LIMIT)
    gnt.gemm_nt_debug_set_fault(fault)
    try:
        _run(A, B, path)
        with pytest.raises(gnt.GemmError) as e:
            gnt.gemm_nt_check()
        assert e.value.status == gnt.Status.DEVICE_TIMEOUT
    finally:
        gnt.gemm_nt_debug_set_fault(0)
        gnt.gemm_nt_debug_set_wait_limit(0)
    gnt.gemm_nt_check()
    out = _run(A, B, path)
    gnt.gemm_nt_check()
    ref, absdot = oracle.gemm_nt(A, B)
    assert_parity(out.cpu().numpy(), ref, absdot, what="after timeout " + path.name)
