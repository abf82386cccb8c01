"""Other instruction shapes: GEMM_PATH_TC05_M64 (64-row tiles on the plain
M = 64 tcgen05.mma) and GEMM_PATH_TC05_WS (32- or 64-row tiles on the
weight-stationary tcgen05.mma.ws, whose accumulator is spread over all 128
TMEM lanes in N/2 or N/4 columns), against the oracle.

Shapes cover one and several row tiles with ragged tails, every tile width
the paths pick (64, 128, 256 columns), the stream-K split for few tiles,
16-bit and 8-bit inputs (packed 4-bit included), 16-bit outputs and the
refusals (block scales, MN-major A)."""
import numpy as np
import pytest

import dense_fp16_tensor_gemm_gb300 as gnt
import gpu_util
import oracle
import workloads
from gpu_util import check_exact, check_tol, run_general

pytestmark = pytest.mark.gpu

P = gnt.Path
SHAPE_PATHS = [P.TC05_M64, P.TC05_WS]


def _inputs(batch, M, N, K, ab, dist="normal", seed=0, sigma=1.0):
    return workloads.make_inputs(batch, M, N, K, dist, sigma, seed=seed, dtype=ab)


@pytest.mark.parametrize("M,N,K", [(1, 70, 64), (31, 130, 200), (32, 520, 1000), (33, 300, 256),
                                   (64, 256, 512), (100, 520, 1000), (300, 130, 384)])
@pytest.mark.parametrize("path", SHAPE_PATHS, ids=lambda p: p.name)
def test_ragged_batched_f16(path, M, N, K):
    A, B = _inputs(2, M, N, K, "f16", seed=M + N + K)
    ref, absdot = oracle.gemm_nt(A, B)
    check_tol(run_general(A, B, "f16", "f32", path), ref, absdot, "f32", "%s %dx%dx%d" % (path.name, M, N, K))


@pytest.mark.parametrize("ab,out", [("bf16", "bf16"), ("e4m3", "f32"), ("e5m2", "f16"), ("e2m1", "f32"),
                                    ("e2m3", "bf16")])
@pytest.mark.parametrize("path", SHAPE_PATHS, ids=lambda p: p.name)
def test_other_types(path, ab, out):
    for M in (20, 90):
        A, B = _inputs(2, M, 300, 384, ab, seed=700 + M)
        ref, absdot = oracle.gemm_nt(A, B, dtype=ab)
        check_tol(run_general(A, B, ab, out, path), ref, absdot, out, "%s M=%d %s->%s" % (path.name, M, ab, out))


@pytest.mark.parametrize("path", SHAPE_PATHS, ids=lambda p: p.name)
def test_integer_inputs_exact(path):
    for M in (24, 200):
        A, B = _inputs(1, M, 700, 1024, "f16", dist="int4", seed=710 + M)
        ref, _ = oracle.gemm_nt(A, B)
        for out in ("f32", "f16", "bf16"):
            check_exact(run_general(A, B, "f16", out, path), ref, out, "%s M=%d ->%s" % (path.name, M, out))


@pytest.mark.parametrize("path", SHAPE_PATHS, ids=lambda p: p.name)
def test_stream_k_long_k(path):
    """Two or four tiles over K = 16384: the iterations are shared by all SMs
    and the pieces of a tile summed with atomics."""
    A, B = _inputs(1, 40, 256, 16384, "f16", seed=720, sigma=0.5)
    ref, absdot = oracle.gemm_nt(A, B)
    check_tol(run_general(A, B, "f16", "f32", path), ref, absdot, "f32", "%s stream-K" % path.name)


@pytest.mark.parametrize("path", SHAPE_PATHS, ids=lambda p: p.name)
def test_b_mn_major_and_refusals(path):
    A, B = _inputs(1, 50, 256, 256, "f16", seed=730)
    ref, absdot = oracle.gemm_nt(A, B)
    check_tol(run_general(A, B, "f16", "f32", path, b_mn=True), ref, absdot, "f32", "%s B MN-major" % path.name)
    with pytest.raises(gnt.GemmError) as e:
        run_general(A, B, "f16", "f32", path, a_mn=True)
    assert e.value.status == gnt.Status.NOT_SUPPORTED
    from test_gpu_mx import draw, run_mx
    A8, SA, B8, SB = draw(1, 50, 256, 256, "e4m3", seed=731)
    with pytest.raises(gnt.GemmError) as e:
        run_mx(A8, SA, B8, SB, "e4m3", "f32", path)
    assert e.value.status == gnt.Status.NOT_SUPPORTED


@pytest.mark.parametrize("path", SHAPE_PATHS, ids=lambda p: p.name)
def test_skinny_64x16384x8192_sampled(path):
    """The skinny workload (M = 64, N = 16384, K = 8192) on these paths, as the
    benchmark runs it with --path; sampled rows, columns and elements."""
    A, B = workloads.workload_inputs("skinny_64x16384x8192")
    got = run_general(A[None], B[None], "f16", "f32", path)
    bb, ii, jj = gpu_util.sample_indices(1, 64, 16384, 4096, rows=(0, 15, 16, 31, 32, -1),
                                         cols=(0, 63, 64, 127, 128, 8191, -1))
    ref, absdot = oracle.gemm_nt_sampled(A[None], B[None], bb, ii, jj)
    check_tol(got[bb, ii, jj], ref, absdot, "f32", "skinny %s" % path.name)
    assert np.isfinite(got).all()
