"""Operands stored K-major or MN-major (gemm_nt_batched_major) on every kernel,
against the oracle.

The oracle computes Out = A @ B.T from the logical operands A (M, K) and
B (N, K); an MN-major operand is handed to the library as its transpose, so
B MN-major is the plain row-major product A @ B' with B' = B.T of shape (K, N)
("NN"), and both MN-major is A'.T @ B' ("TN").  The warp kernel reads an
MN-major tile with ldmatrix's .trans form ("Warp Matrix Instructions", "Other
Fragment Shapes and Transfers"; "copy -> ldstmatrix", "Algorithm" step 3); the
tcgen05 kernels with MN-major shared-memory descriptors.
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
# (a_mn, b_mn) with readable ids: "aK-bMN" is NN, "aMN-bMN" is TN
MAJORS = [(False, True), (True, False), (True, True), (False, False)]
MAJOR_IDS = ["a%s-b%s" % ("MN" if a else "K", "MN" if b else "K") for a, b in MAJORS]


def _inputs(batch, M, N, K, ab="f16", dist="normal", seed=0):
    return workloads.make_inputs(batch, M, N, K, dist, 1.0, seed=seed, dtype=ab)


@pytest.mark.parametrize("path", [P.AUTO, P.TC05, P.TC05_PAIR, P.MMASYNC], ids=lambda p: p.name)
@pytest.mark.parametrize("a_mn,b_mn", MAJORS, ids=MAJOR_IDS)
def test_ragged_batched(a_mn, b_mn, path):
    """Several tiles in each direction, ragged M/N/K tails, batch 2."""
    A, B = _inputs(2, 300, 520, 264, seed=201)
    ref, absdot = oracle.gemm_nt(A, B)
    got = run_general(A, B, "f16", "f32", path, a_mn, b_mn)
    check_tol(got, ref, absdot, "f32", "%s a_mn=%d b_mn=%d" % (path.name, a_mn, b_mn))


@pytest.mark.parametrize("path", [P.TC05, P.TC05_PAIR, P.MMASYNC, P.SKINNY], ids=lambda p: p.name)
@pytest.mark.parametrize("a_mn,b_mn", MAJORS, ids=MAJOR_IDS)
def test_integer_inputs_bit_exact(a_mn, b_mn, path):
    M = 48 if path == P.SKINNY else 200
    A, B = _inputs(1, M, 1100, 1000, dist="int4", seed=202)
    ref, _ = oracle.gemm_nt(A, B)
    check_exact(run_general(A, B, "f16", "f32", path, a_mn, b_mn), ref, "f32",
                "%s a_mn=%d b_mn=%d" % (path.name, a_mn, b_mn))


@pytest.mark.parametrize("M,N,K", [(1, 1024, 64), (33, 1500, 1000), (64, 4096, 520), (64, 16384, 512)])
@pytest.mark.parametrize("a_mn,b_mn", MAJORS[:3], ids=MAJOR_IDS[:3])
def test_skinny(a_mn, b_mn, M, N, K):
    """The swapped kernel: X = B (MN-major when B is), Y = A; a long N takes
    tiles or stream-K instead of the K-major row split when B is MN-major."""
    A, B = _inputs(1, M, N, K, seed=M + N + K)
    ref, absdot = oracle.gemm_nt(A, B)
    check_tol(run_general(A, B, "f16", "f32", P.SKINNY, a_mn, b_mn), ref, absdot, "f32",
              "SKINNY %dx%dx%d a_mn=%d b_mn=%d" % (M, N, K, a_mn, b_mn))


@pytest.mark.parametrize("out", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("path", [P.AUTO, P.TC05, P.TC05_PAIR, P.MMASYNC], ids=lambda p: p.name)
def test_bf16_and_16_bit_outputs(path, out):
    A, B = _inputs(2, 260, 390, 200, ab="bf16", seed=203)
    ref, absdot = oracle.gemm_nt(A, B, dtype="bf16")
    for a_mn, b_mn in MAJORS[:3]:
        check_tol(run_general(A, B, "bf16", out, path, a_mn, b_mn), ref, absdot, out,
                  "%s bf16->%s a_mn=%d b_mn=%d" % (path.name, out, a_mn, b_mn))


@pytest.mark.parametrize("a_mn,b_mn", MAJORS[:3], ids=MAJOR_IDS[:3])
def test_padded_pitches(a_mn, b_mn):
    """Row pitches beyond the stored rows: multiples of 8 keep the tensor-core
    kernels; an odd pitch moves to the warp kernel."""
    A, B = _inputs(1, 300, 270, 200, seed=204)
    ref, absdot = oracle.gemm_nt(A, B)
    lda = (304 if a_mn else 200) + 24   # stored row lengths rounded up to 8, plus padding
    ldb = (272 if b_mn else 200) + 40
    for path in (P.AUTO, P.TC05, P.TC05_PAIR, P.MMASYNC):
        check_tol(run_general(A, B, "f16", "f32", path, a_mn, b_mn, lda=lda, ldb=ldb), ref, absdot, "f32",
                  "%s padded" % path.name)
    check_tol(run_general(A, B, "f16", "f32", P.AUTO, a_mn, b_mn, lda=lda + 1, ldb=ldb + 3), ref, absdot,
              "f32", "odd pitches")
    with pytest.raises(gnt.GemmError) as e:
        run_general(A, B, "f16", "f32", P.TC05, a_mn, b_mn, lda=lda + 1, ldb=ldb + 3)
    assert e.value.status == gnt.Status.NOT_SUPPORTED


def test_misaligned_base_uses_warp_kernel():
    import torch
    A, B = _inputs(1, 150, 140, 136, seed=205)
    ref, absdot = oracle.gemm_nt(A, B)
    check_tol(run_general(A, B, "f16", "f32", P.AUTO, True, True, a_offset=1), ref, absdot, "f32", "offset A")
    a = torch.zeros(136 * 150 + 1, dtype=torch.float16, device="cuda")
    b = torch.zeros(136 * 140, dtype=torch.float16, device="cuda")
    o = torch.zeros(150 * 140, dtype=torch.float32, device="cuda")
    with pytest.raises(gnt.GemmError) as e:
        gnt.gemm_nt_batched_major(a.data_ptr() + 2, gnt.Major.MN, b.data_ptr(), gnt.Major.MN, o.data_ptr(),
                                  gnt.DType.F16, gnt.DType.F32, 150, 140, 136, 150, 140, 140, 0, 0, 0, 1,
                                  P.TC05_PAIR, torch.cuda.current_stream().cuda_stream)
    assert e.value.status == gnt.Status.NOT_SUPPORTED


@pytest.mark.parametrize("a_mn,b_mn", MAJORS[:3], ids=MAJOR_IDS[:3])
def test_shared_operand(a_mn, b_mn):
    """Batch stride 0 on an MN-major operand: every batch reuses it."""
    import torch
    batch, M, N, K = 3, 200, 300, 136
    A, B1 = _inputs(batch, M, N, K, seed=206)
    B = np.repeat(B1[:1], batch, axis=0)
    ref, absdot = oracle.gemm_nt(A, B)
    As = np.ascontiguousarray(np.swapaxes(A, 1, 2)) if a_mn else A
    Bs = np.ascontiguousarray(np.swapaxes(B1[:1], 1, 2)) if b_mn else B1[:1]
    a, pa = gpu_util.to_device(As, "f16")
    b, pb = gpu_util.to_device(Bs, "f16")
    o = torch.full((batch, M, N), float("nan"), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    gnt.gemm_nt_batched_major(pa, gnt.Major.MN if a_mn else gnt.Major.K, pb, gnt.Major.MN if b_mn else gnt.Major.K,
                              o.data_ptr(), gnt.DType.F16, gnt.DType.F32, M, N, K, As.shape[2], Bs.shape[2], N,
                              As.shape[1] * As.shape[2], 0, M * N, batch, P.AUTO, stream)
    gnt.gemm_nt_check(stream)
    check_tol(o.double().cpu().numpy(), ref, absdot, "f32", "shared B")


@pytest.mark.parametrize("a_mn,b_mn", MAJORS[:3], ids=MAJOR_IDS[:3])
def test_long_k_few_tiles(a_mn, b_mn):
    """Few tiles and a long K: the pair kernel's split-K fixup and the one-CTA
    kernel's stream-K run on MN-major operands."""
    A, B = _inputs(1, 512, 512, 8192, seed=207)
    ref, absdot = oracle.gemm_nt(A, B)
    for path in (P.AUTO, P.TC05):
        check_tol(run_general(A, B, "f16", "f32", path, a_mn, b_mn), ref, absdot, "f32",
                  "%s long K a_mn=%d b_mn=%d" % (path.name, a_mn, b_mn))


def test_nn_product_of_row_major_matrices():
    """The plain row-major product C = X @ Y with X (M, K) and Y (K, N) is the
    call with A = X (K-major) and B given as Y (MN-major)."""
    import torch
    M, K, N = 384, 320, 448
    X, Yt = _inputs(1, M, N, K, seed=208)
    Y = np.ascontiguousarray(Yt[0].T)  # (K, N) row-major
    ref, absdot = oracle.gemm_nt(X[0], np.ascontiguousarray(Y.T))
    x, y = gpu_util.to_device(X, "f16")[0], gpu_util.to_device(Y[None], "f16")[0]
    c = torch.empty((M, N), dtype=torch.float32, device="cuda")
    gnt.gemm_nt_batched_major(x.data_ptr(), gnt.Major.K, y.data_ptr(), gnt.Major.MN, c.data_ptr(), gnt.DType.F16,
                              gnt.DType.F32, M, N, K, K, N, N, 0, 0, 0, 1, P.AUTO,
                              torch.cuda.current_stream().cuda_stream)
    gnt.gemm_nt_check()
    check_tol(c.double().cpu().numpy(), ref, absdot, "f32", "NN")
