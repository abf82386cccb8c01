"""6- and 4-bit float inputs (E2M3, E3M2, E2M1), packed along K, on the
tcgen05 kernels, plain and block-scaled, against the oracle.

The library takes them packed (fp4 two per byte, fp6 four per three bytes,
little-endian bit order); its tensor maps spread every 16 packed elements to
a 16-byte chunk of shared memory, the layout kind::f8f6f4 reads them in, so the
stages and MMAs are those of the 8-bit floats with the format codes 3, 4, 5 in
the instruction descriptor.  The oracle takes the same codes one per element;
the tests pack them for the device (workloads.pack_subbyte), so parity also
checks the packing.  Products of two such values are exact in fp32; integer
inputs are exact on every path."""
import numpy as np
import pytest

import dense_fp16_tensor_gemm_gb300 as gnt
import oracle
import workloads
from gpu_util import check_exact, check_tol, run_general
from test_gpu_mx import draw, run_mx

pytestmark = pytest.mark.gpu

P = gnt.Path
F6F4 = ["e2m3", "e3m2", "e2m1"]


def _inputs(batch, M, N, K, ab, dist="normal", seed=0, sigma=1.0):
    return workloads.make_inputs(batch, M, N, K, dist, sigma, seed=seed, dtype=ab)


@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("ab", F6F4)
@pytest.mark.parametrize("path", [P.AUTO, P.TC05, P.TC05_PAIR], ids=lambda p: p.name)
def test_ragged_batched(path, ab, out):
    """Several tiles each way, ragged M and N, K = 384, batch 2."""
    A, B = _inputs(2, 300, 520, 384, ab, seed=601)
    ref, absdot = oracle.gemm_nt(A, B, dtype=ab)
    check_tol(run_general(A, B, ab, out, path), ref, absdot, out, "%s %s->%s" % (path.name, ab, out))


@pytest.mark.parametrize("ab", F6F4)
@pytest.mark.parametrize("path", [P.TC05, P.TC05_PAIR, P.SKINNY], ids=lambda p: p.name)
def test_integer_inputs_exact(path, ab):
    M = 48 if path == P.SKINNY else 200
    A, B = _inputs(1, M, 1100, 1024, ab, dist="int4", seed=602)
    ref, _ = oracle.gemm_nt(A, B, dtype=ab)
    for out in ("f32", "f16", "bf16"):
        check_exact(run_general(A, B, ab, out, path), ref, out, "%s %s->%s" % (path.name, ab, out))


@pytest.mark.parametrize("ab", F6F4)
@pytest.mark.parametrize("M,N,K", [(1, 1024, 128), (33, 1500, 1152), (64, 16384, 1024)])
def test_skinny(M, N, K, ab):
    A, B = _inputs(1, M, N, K, ab, seed=M + N + K, sigma=0.5)
    ref, absdot = oracle.gemm_nt(A, B, dtype=ab)
    check_tol(run_general(A, B, ab, "f32", P.AUTO), ref, absdot, "f32", "skinny %dx%dx%d %s" % (M, N, K, ab))


@pytest.mark.parametrize("ab", F6F4)
def test_padded_pitch_and_refusals(ab):
    """A pitch of K + 128 elements runs; a K that is not a multiple of 128, a
    pitch of a few bytes more, or the warp kernel are refused with
    NOT_SUPPORTED, and an MN-major packed operand with INVALID_VALUE."""
    A, B = _inputs(1, 260, 300, 256, ab, seed=603)
    ref, absdot = oracle.gemm_nt(A, B, dtype=ab)
    check_tol(run_general(A, B, ab, "f32", P.AUTO, lda=384, ldb=384), ref, absdot, "f32", "pitch K+128")
    A2, B2 = _inputs(1, 260, 300, 200, ab, seed=604)
    for args in ((A2, B2, ab, "f32", P.AUTO), (A, B, ab, "f32", P.AUTO, False, False, 260, 260),
                 (A, B, ab, "f32", P.MMASYNC)):
        with pytest.raises(gnt.GemmError) as e:
            run_general(*args)
        assert e.value.status == gnt.Status.NOT_SUPPORTED
    import torch
    z = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    o = torch.zeros(260 * 300, dtype=torch.float32, device="cuda")
    with pytest.raises(gnt.GemmError) as e:
        gnt.gemm_nt_batched_major(z.data_ptr(), gnt.Major.MN, z.data_ptr() + 65536, gnt.Major.K, o.data_ptr(),
                                  getattr(gnt.DType, ab.upper()), gnt.DType.F32, 260, 300, 256, 260, 256, 300,
                                  0, 0, 0, 1, P.AUTO, torch.cuda.current_stream().cuda_stream)
    assert e.value.status == gnt.Status.INVALID_VALUE


@pytest.mark.parametrize("ab", F6F4)
@pytest.mark.parametrize("path", [P.AUTO, P.TC05, P.TC05_PAIR, P.SKINNY], ids=lambda p: p.name)
def test_block_scaled(path, ab):
    M = 48 if path == P.SKINNY else 300
    A, SA, B, SB = draw(2, M, 1100, 384, ab, seed=606)
    ref, absdot = oracle.gemm_nt_mx(A, SA, B, SB, dtype=ab)
    check_tol(run_mx(A, SA, B, SB, ab, "f32", path), ref, absdot, "f32", "%s mx %s" % (path.name, ab))


@pytest.mark.parametrize("ab", F6F4)
def test_block_scaled_integers_exact(ab):
    A, SA, B, SB = draw(1, 256, 640, 1024, ab, dist="int4", seed=607, lo=124, hi=131)
    ref, _ = oracle.gemm_nt_mx(A, SA, B, SB, dtype=ab)
    check_exact(run_mx(A, SA, B, SB, ab, "f32", P.AUTO), ref, "f32", "mx integers %s" % ab)


@pytest.mark.parametrize("ab,mx", [("e2m1", False), ("e2m3", False), ("e2m1", True), ("e3m2", True)])
def test_square_8192_sampled(ab, mx):
    """The 8192^3 workload's draws rounded to the type, as the benchmark runs
    it (its block scales for the block-scaled product), on the path it takes;
    sampled rows and columns across tile edges and random elements."""
    import gpu_util
    A, B = workloads.workload_inputs("square_8192", ab)
    A3, B3 = A[None], B[None]
    if mx:
        SA, SB = workloads.workload_mx_scales("square_8192")
        got = run_mx(A3, SA[None], B3, SB[None], ab, "f32", P.AUTO)
    else:
        got = run_general(A3, B3, ab, "f32", P.AUTO)
    bb, ii, jj = gpu_util.sample_indices(1, 8192, 8192, 4096, rows=(0, 127, 128, 4095, -1), cols=(0, 255, 256, -1))
    if mx:
        ref, absdot = oracle.gemm_nt_sampled_mx(A3, SA[None], B3, SB[None], bb, ii, jj, dtype=ab)
    else:
        ref, absdot = oracle.gemm_nt_sampled(A3, B3, bb, ii, jj, dtype=ab)
    check_tol(got[bb, ii, jj], ref, absdot, "f32", "square_8192 %s%s" % (ab, " mx" if mx else ""))


@pytest.mark.parametrize("ab", F6F4)
def test_torch_binding(ab):
    """gemm_nt_packed on uint8 tensors of packed rows, plain and block-scaled,
    and its argument checks."""
    import torch
    code = getattr(gnt.DType, ab.upper())
    A, B = _inputs(1, 130, 250, 256, ab, seed=608)
    a = torch.from_numpy(workloads.pack_subbyte(A[0], ab)).cuda()
    b = torch.from_numpy(workloads.pack_subbyte(B[0], ab)).cuda()
    ref, absdot = oracle.gemm_nt(A, B, dtype=ab)
    out = gnt.gemm_nt_packed(a, b, 256, code)
    check_tol(out.double().cpu().numpy()[None], ref, absdot, "f32", "gemm_nt_packed %s" % ab)
    rng = np.random.default_rng(609)
    SA = rng.integers(122, 133, size=(130, 8)).astype(np.uint8)
    SB = rng.integers(122, 133, size=(250, 8)).astype(np.uint8)
    ref, absdot = oracle.gemm_nt_mx(A, SA[None], B, SB[None], dtype=ab)
    out = gnt.gemm_nt_packed(a, b, 256, code, torch.from_numpy(SA).cuda(), torch.from_numpy(SB).cuda(),
                             out_dtype=torch.bfloat16)
    check_tol(out.double().cpu().numpy()[None], ref, absdot, "bf16", "gemm_nt_packed mx %s" % ab)
    with pytest.raises(ValueError):
        gnt.gemm_nt_packed(a, b, 128, code)  # rows hold 256 elements
    with pytest.raises(TypeError):
        gnt.gemm_nt_packed(a.view(torch.int8), b, 256, code)
    with pytest.raises(TypeError):
        gnt.gemm_nt_packed(a, b, 256, gnt.DType.E4M3)
    with pytest.raises(ValueError):
        gnt.gemm_nt_packed(a, b, 256, code, torch.from_numpy(SA).cuda())
    torch.cuda.synchronize()
