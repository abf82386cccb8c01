"""8-bit float inputs (E4M3, E5M2) on every kernel, against the oracle.

The tcgen05 kernels run them on kind::f8f6f4 (a stage row of 128 bytes holds
128 elements of K, four 32-wide MMAs per stage); the warp kernel widens them
to fp16 while staging, which is exact.  Products of two 8-bit values are exact
in fp32, so the parity bound is the fp16 one, plus the output rounding of a
16-bit Out; integer inputs are exact on every path.
"""
import numpy as np
import pytest

import dense_fp16_tensor_gemm_gb300 as gnt
import gpu_util
import oracle
import workloads
from gpu_util import check_exact, check_tol, run_general

pytestmark = pytest.mark.gpu

P = gnt.Path
F8 = ["e4m3", "e5m2"]


def _inputs(batch, M, N, K, ab, dist="normal", seed=0, sigma=1.0):
    return workloads.make_inputs(batch, M, N, K, dist, sigma, seed=seed, dtype=ab)


@pytest.mark.parametrize("out", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("ab", F8)
@pytest.mark.parametrize("path", [P.AUTO, P.TC05, P.TC05_PAIR, P.MMASYNC], ids=lambda p: p.name)
def test_ragged_batched(path, ab, out):
    """Several tiles each way, ragged M and N, and K = 400 (three 128-wide
    stages and a 16-element tail), batch 2."""
    A, B = _inputs(2, 300, 520, 400, ab, seed=301)
    ref, absdot = oracle.gemm_nt(A, B, dtype=ab)
    check_tol(run_general(A, B, ab, out, path), ref, absdot, out, "%s %s->%s" % (path.name, ab, out))


@pytest.mark.parametrize("ab", F8)
@pytest.mark.parametrize("path", [P.TC05, P.TC05_PAIR, P.SKINNY, P.MMASYNC], ids=lambda p: p.name)
def test_integer_inputs_exact(path, ab):
    M = 48 if path == P.SKINNY else 200
    A, B = _inputs(1, M, 1100, 1008, ab, dist="int4", seed=302)
    ref, _ = oracle.gemm_nt(A, B, dtype=ab)
    for out in ("f32", "f16", "bf16"):
        check_exact(run_general(A, B, ab, out, path), ref, out, "%s %s->%s" % (path.name, ab, out))


@pytest.mark.parametrize("ab", F8)
@pytest.mark.parametrize("M,N,K", [(1, 1024, 128), (33, 1500, 1024), (64, 4096, 528), (64, 16384, 1024)])
def test_skinny(M, N, K, ab):
    A, B = _inputs(1, M, N, K, ab, seed=M + N + K, sigma=0.5)
    ref, absdot = oracle.gemm_nt(A, B, dtype=ab)
    check_tol(run_general(A, B, ab, "f32", P.SKINNY), ref, absdot, "f32", "SKINNY %dx%dx%d %s" % (M, N, K, ab))


@pytest.mark.parametrize("ab", F8)
def test_layouts_off_the_tensor_cores(ab):
    """Pitches that are not multiples of 16 bytes, an odd base and MN-major
    operands run on the warp kernel; the tensor-core paths refuse them."""
    A, B = _inputs(1, 150, 140, 136, ab, seed=303)
    ref, absdot = oracle.gemm_nt(A, B, dtype=ab)
    check_tol(run_general(A, B, ab, "f32", P.AUTO, lda=160, ldb=144), ref, absdot, "f32", "pitch 160/144")
    check_tol(run_general(A, B, ab, "f32", P.AUTO, lda=139, ldb=141), ref, absdot, "f32", "odd pitches")
    check_tol(run_general(A, B, ab, "f32", P.AUTO, a_offset=3), ref, absdot, "f32", "odd base")
    for a_mn, b_mn in ((False, True), (True, False), (True, True)):
        check_tol(run_general(A, B, ab, "bf16", P.AUTO, a_mn, b_mn), ref, absdot, "bf16",
                  "a_mn=%d b_mn=%d" % (a_mn, b_mn))
        with pytest.raises(gnt.GemmError) as e:
            run_general(A, B, ab, "f32", P.TC05, a_mn, b_mn)
        assert e.value.status == gnt.Status.NOT_SUPPORTED
    with pytest.raises(gnt.GemmError) as e:
        run_general(A, B, ab, "f32", P.TC05_PAIR, lda=139, ldb=141)
    assert e.value.status == gnt.Status.NOT_SUPPORTED


def test_long_k_split_and_e5m2_range():
    """Few tiles and K = 16384 (128 stages): the pair kernel splits K across
    pairs; E5M2 values up to +-4096 (normal(0, 1000)) exercise its range."""
    A, B = _inputs(1, 512, 512, 16384, "e5m2", seed=304, sigma=1000.0)
    ref, absdot = oracle.gemm_nt(A, B, dtype="e5m2")
    check_tol(run_general(A, B, "e5m2", "f32", P.AUTO), ref, absdot, "f32", "split")
    check_tol(run_general(A, B, "e5m2", "f32", P.TC05), ref, absdot, "f32", "one CTA per tile")


def test_torch_wrapper_and_square_sample():
    import torch
    A, B = _inputs(0, 1024, 768, 512, "e4m3", seed=305)
    ref, absdot = oracle.gemm_nt(A, B, dtype="e4m3")
    a = torch.from_numpy(A.copy()).view(torch.float8_e4m3fn).cuda()
    b = torch.from_numpy(B.copy()).view(torch.float8_e4m3fn).cuda()
    out = gnt.gemm_nt(a, b)
    assert out.dtype == torch.float32
    check_tol(out.double().cpu().numpy()[None], ref[None], absdot[None], "f32", "wrapper")
    out16 = gnt.gemm_nt(a, b, out_dtype=torch.bfloat16)
    check_tol(out16.double().cpu().numpy()[None], ref[None], absdot[None], "bf16", "wrapper bf16")
    with pytest.raises(TypeError):
        gnt.gemm_nt(a, b.view(torch.float8_e5m2))


def test_square_4096_sampled():
    """The square 4096 recipe (uniform[-1,1], seed 1) in E4M3, sampled rows,
    columns and random elements."""
    w = workloads.WORKLOADS["square_4096"]
    A, B = workloads.make_inputs(1, w.M, w.N, w.K, w.dist, w.sigma, w.seed, dtype="e4m3")
    got = run_general(A, B, "e4m3", "f32", P.AUTO)
    bb, ii, jj = gpu_util.sample_indices(1, w.M, w.N, 4000, rows=(0, 255, 256, -1), cols=(0, 255, -1))
    ref, absdot = oracle.gemm_nt_sampled(A, B, bb, ii, jj, dtype="e4m3")
    check_tol(got[bb, ii, jj], ref, absdot, "f32", "square_4096 e4m3")
