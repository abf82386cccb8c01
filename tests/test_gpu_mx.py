"""Block-scaled 8-bit products (gemm_nt_mx): E4M3 / E5M2 inputs with one E8M0
scale per 32 consecutive K elements of every row, on the tcgen05
kind::mxf8f6f4 kernels, against the oracle's gemm_nt_mx.

Scales are drawn as plain (rows, ceil(K/32)) bytes, packed on the device by
the library (checked here against a numpy packing of the layout the header
defines), and the same plain scales go to the oracle."""
import numpy as np
import pytest

import dense_fp16_tensor_gemm_gb300 as gnt
import gpu_util
import oracle
import workloads
from gpu_util import check_exact, check_tol

pytestmark = pytest.mark.gpu

P = gnt.Path
F8 = ["e4m3", "e5m2"]


def pack_ref(S, K):
    """numpy packing of plain scales (batch, rows, ceil(K/32)) into the atom
    layout: byte 16*r + 4*q + s of atom (rb, kg) = S[rb*128 + 32*q + r, 4*kg + s]."""
    batch, rows, kb = S.shape
    RB, KG = (rows + 127) // 128, (K + 127) // 128
    pad = np.full((batch, RB * 128, KG * 4), 127, dtype=np.uint8)
    pad[:, :rows, :kb] = S
    return np.ascontiguousarray(pad.reshape(batch, RB, 4, 32, KG, 4).transpose(0, 1, 4, 3, 2, 5)).reshape(-1)


def draw(batch, M, N, K, ab, dist="normal", seed=0, sigma=1.0, lo=118, hi=137):
    A, B = workloads.make_inputs(batch, M, N, K, dist, sigma, seed=seed, dtype=ab)
    rng = np.random.default_rng(seed + 1000)
    kb = (K + 31) // 32
    SA = rng.integers(lo, hi, size=(batch, M, kb)).astype(np.uint8)
    SB = rng.integers(lo, hi, size=(batch, N, kb)).astype(np.uint8)
    return A, SA, B, SB


def run_mx(A, SA, B, SB, ab, out, path, shared_b=False, lda=None, pack_on_host=False):
    """Out through gemm_nt_mx; scales packed by the library (or by pack_ref).
    Returns float64 (batch, M, N)."""
    import torch
    batch, M, K = A.shape
    N = B.shape[1]
    lda = lda or K
    if ab in gpu_util.PACKED:
        a, pa = gpu_util.to_device_packed(A, ab, lda)
        b, pb = gpu_util.to_device_packed(B[:1] if shared_b else B, ab, K)
    else:
        a, pa = gpu_util.to_device(A, ab, lda)
        b, pb = gpu_util.to_device(B[:1] if shared_b else B, ab)
    SBu = SB[:1] if shared_b else SB
    if pack_on_host:
        sa = torch.from_numpy(pack_ref(SA, K)).cuda()
        sb = torch.from_numpy(pack_ref(SBu, K)).cuda()
    else:
        sa = gnt.pack_mx_scales(torch.from_numpy(SA).cuda(), K)
        sb = gnt.pack_mx_scales(torch.from_numpy(SBu).cuda(), K)
    o = torch.full((batch, M, N), float("nan"), dtype=gpu_util.torch_dtype(out), device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    gnt.gemm_nt_mx(pa, sa.data_ptr(), pb, sb.data_ptr(), o.data_ptr(), gpu_util.dtype_code(ab),
                   gpu_util.dtype_code(out), M, N, K, lda, K, N, M * lda, 0 if shared_b else N * K, M * N, batch,
                   path, stream)
    gnt.gemm_nt_check(stream)
    return o.double().cpu().numpy()


def test_pack_matches_the_layout():
    import torch
    rng = np.random.default_rng(501)
    for (batch, rows, K) in ((1, 1, 32), (2, 300, 400), (1, 128, 128), (3, 129, 1000)):
        S = rng.integers(0, 255, size=(batch, rows, (K + 31) // 32)).astype(np.uint8)
        got = gnt.pack_mx_scales(torch.from_numpy(S).cuda(), K).cpu().numpy()
        assert got.size == batch * gnt.gemm_nt_mx_scale_bytes(rows, K)
        assert np.array_equal(got, pack_ref(S, K)), (batch, rows, K)


@pytest.mark.parametrize("out", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("ab", F8)
@pytest.mark.parametrize("path", [P.AUTO, P.TC05, P.TC05_PAIR], ids=lambda p: p.name)
def test_ragged_batched(path, ab, out):
    """Several tiles each way, ragged M and N, K = 400 (three 128-element
    stages, a 16-element tail, a partial 32-element scale block), batch 2."""
    # fp16 Out holds at most 65504: keep its sums in range with scales <= 1
    A, SA, B, SB = draw(2, 300, 520, 400, ab, seed=502, hi=128 if out == "f16" else 137)
    ref, absdot = oracle.gemm_nt_mx(A, SA, B, SB, dtype=ab)
    if out == "f16":
        assert np.abs(ref).max() < 60000
    check_tol(run_mx(A, SA, B, SB, ab, out, path), ref, absdot, out, "%s %s->%s" % (path.name, ab, out))


@pytest.mark.parametrize("ab", F8)
@pytest.mark.parametrize("path", [P.TC05, P.SKINNY, P.TC05_PAIR], ids=lambda p: p.name)
def test_integer_inputs_exact(path, ab):
    """Integers in [-4, 4] and scales 2^-3..2^3: every partial sum is exact."""
    M = 48 if path == P.SKINNY else 200
    A, SA, B, SB = draw(1, M, 1100, 1008, ab, dist="int4", seed=503, lo=124, hi=131)
    ref, _ = oracle.gemm_nt_mx(A, SA, B, SB, dtype=ab)
    for out in ("f32", "bf16"):
        check_exact(run_mx(A, SA, B, SB, ab, out, path), ref, out, "%s %s->%s" % (path.name, ab, out))


@pytest.mark.parametrize("ab", F8)
@pytest.mark.parametrize("M,N,K", [(1, 1024, 128), (33, 1500, 1056), (64, 16384, 1024), (64, 4096, 528)])
def test_skinny(M, N, K, ab):
    A, SA, B, SB = draw(1, M, N, K, ab, seed=M + N + K, sigma=0.5)
    ref, absdot = oracle.gemm_nt_mx(A, SA, B, SB, dtype=ab)
    check_tol(run_mx(A, SA, B, SB, ab, "f32", P.AUTO), ref, absdot, "f32", "skinny %dx%dx%d %s" % (M, N, K, ab))


def test_host_packed_scales_and_wide_scale_range():
    """Scales packed by the numpy reference, spread over 2^-40..2^40."""
    A, SA, B, SB = draw(1, 256, 384, 768, "e4m3", seed=504, lo=87, hi=168)
    ref, absdot = oracle.gemm_nt_mx(A, SA, B, SB, dtype="e4m3")
    check_tol(run_mx(A, SA, B, SB, "e4m3", "f32", P.TC05, pack_on_host=True), ref, absdot, "f32", "wide scales")


def test_shared_operand_and_padded_pitch():
    """B (and its scales) shared by every batch (stride 0); A with a padded
    row pitch."""
    A, SA, B1, SB1 = draw(3, 200, 300, 512, "e5m2", seed=505)
    B = np.repeat(B1[:1], 3, axis=0)
    SB = np.repeat(SB1[:1], 3, axis=0)
    ref, absdot = oracle.gemm_nt_mx(A, SA, B, SB, dtype="e5m2")
    check_tol(run_mx(A, SA, B, SB, "e5m2", "f32", P.AUTO, shared_b=True, lda=544), ref, absdot, "f32", "shared B")


@pytest.mark.parametrize("path", [P.TC05, P.TC05_PAIR], ids=lambda p: p.name)
def test_long_k_few_tiles(path):
    """Few tiles and K = 16384: both kernels split K (stream-K; the pair
    kernel through its workspace slices)."""
    A, SA, B, SB = draw(1, 256, 256, 16384, "e4m3", seed=506, sigma=0.25)
    ref, absdot = oracle.gemm_nt_mx(A, SA, B, SB, dtype="e4m3")
    check_tol(run_mx(A, SA, B, SB, "e4m3", "f32", path), ref, absdot, "f32", "stream-K")


@pytest.mark.parametrize("M,N,K", [(256, 192, 128), (640, 1000, 384), (1000, 576, 256), (130, 1300, 640)])
def test_pair_tile_windows(M, N, K):
    """Pair tiles over ragged M and N: Out rows 32-byte aligned (N a multiple
    of 8) run 256 x 256 tiles with one accumulator, N = 1300 the 256 x 192
    tiles, whose B rows start 0 or 64 rows into a 128-row scale atom."""
    A, SA, B, SB = draw(1, M, N, K, "e5m2", seed=M + N + K)
    ref, absdot = oracle.gemm_nt_mx(A, SA, B, SB, dtype="e5m2")
    check_tol(run_mx(A, SA, B, SB, "e5m2", "f32", P.TC05_PAIR), ref, absdot, "f32", "pair %dx%dx%d" % (M, N, K))


@pytest.mark.parametrize("batch,M,N,K,ab,shared", [(1, 300, 96, 384, "e4m3", False), (3, 200, 264, 512, "e4m3", False),
                                                    (2, 260, 264, 256, "e5m2", True), (2, 257, 520, 640, "e2m1", False)])
def test_single_accumulator_scale_boxes(batch, M, N, K, ab, shared):
    """256 x 256 pair tiles (Out rows 32-byte aligned) take B's scale atoms in
    each data stage, four times over: N = 96 (one row block, a box of one),
    batches whose B row blocks follow one another in the packed scales, B and
    its scales shared by every batch, and packed 4-bit elements.  Integer
    inputs and scales 2^-3..2^3 make every result exact."""
    A, SA, B, SB = draw(batch, M, N, K, ab, dist="int4", seed=507 + N, lo=124, hi=131)
    if shared:
        B = np.repeat(B[:1], batch, axis=0)
        SB = np.repeat(SB[:1], batch, axis=0)
    ref, _ = oracle.gemm_nt_mx(A, SA, B, SB, dtype=ab)
    out = run_mx(A, SA, B, SB, ab, "f32", P.TC05_PAIR, shared_b=shared)
    check_exact(out, ref, "f32", "pair %d x %dx%dx%d %s%s" % (batch, M, N, K, ab, " shared B" if shared else ""))


def test_unit_scales_equal_the_unscaled_product():
    """Scales of 127 on the device give the unscaled 8-bit kernel's result
    (both fp32-accumulated, compared through the oracle)."""
    A, SA, B, SB = draw(1, 300, 260, 640, "e4m3", seed=507, lo=127, hi=128)
    ref, absdot = oracle.gemm_nt(A, B, dtype="e4m3")
    check_tol(run_mx(A, SA, B, SB, "e4m3", "f32", P.AUTO), ref, absdot, "f32", "unit scales")


def test_torch_wrapper_and_unsupported_paths():
    import torch
    A, SA, B, SB = draw(0 + 1, 192, 256, 320, "e4m3", seed=508)
    ref, absdot = oracle.gemm_nt_mx(A[0], SA[0], B[0], SB[0], dtype="e4m3")
    a = torch.from_numpy(A[0].copy()).view(torch.float8_e4m3fn).cuda()
    b = torch.from_numpy(B[0].copy()).view(torch.float8_e4m3fn).cuda()
    sa, sb = torch.from_numpy(SA[0]).cuda(), torch.from_numpy(SB[0]).cuda()
    out = gnt.gemm_nt_mx_tensors(a, sa, b, sb)
    check_tol(out.double().cpu().numpy(), ref, absdot, "f32", "wrapper")
    out16 = gnt.gemm_nt_mx_tensors(a, sa, b, sb, out_dtype=torch.bfloat16)
    check_tol(out16.double().cpu().numpy(), ref, absdot, "bf16", "wrapper bf16")
    pa, pb = gnt.pack_mx_scales(sa, 320), gnt.pack_mx_scales(sb, 320)
    o = torch.empty((192, 256), dtype=torch.float32, device="cuda")
    for path in (P.MMASYNC,):
        with pytest.raises(gnt.GemmError) as e:
            gnt.gemm_nt_mx(a.data_ptr(), pa.data_ptr(), b.data_ptr(), pb.data_ptr(), o.data_ptr(), gnt.DType.E4M3,
                           gnt.DType.F32, 192, 256, 320, 320, 320, 256, 0, 0, 0, 1, path,
                           torch.cuda.current_stream().cuda_stream)
        assert e.value.status == gnt.Status.NOT_SUPPORTED
    # a pitch that is not a multiple of 16 bytes: no block-scaled kernel reads it
    A, SA, B, SB = draw(1, 64, 512, 520, "e4m3", seed=509)
    with pytest.raises(gnt.GemmError) as e:
        run_mx(A, SA, B, SB, "e4m3", "f32", P.AUTO)
    assert e.value.status == gnt.Status.NOT_SUPPORTED


@pytest.mark.parametrize("ab", ["e4m3", "e2m1"])
def test_skinny_workload_sampled(ab):
    """The skinny workload (64 x 16384 x 8192) block-scaled, with its scales, as
    the benchmark runs it (whole 128-row tiles of B on the swapped kernel);
    sampled rows, columns and random elements."""
    A, B = workloads.workload_inputs("skinny_64x16384x8192", ab)
    SA, SB = workloads.workload_mx_scales("skinny_64x16384x8192")
    got = run_mx(A[None], SA[None], B[None], SB[None], ab, "f32", P.AUTO)
    bb, ii, jj = gpu_util.sample_indices(1, 64, 16384, 4096, rows=(0, 31, 32, -1), cols=(0, 127, 128, 8191, -1))
    ref, absdot = oracle.gemm_nt_sampled_mx(A[None], SA[None], B[None], SB[None], bb, ii, jj, dtype=ab)
    check_tol(got[bb, ii, jj], ref, absdot, "f32", "skinny workload mx %s" % ab)


@pytest.mark.parametrize("M,N,K", [(640, 1000, 384), (300, 2000, 1152)])
@pytest.mark.parametrize("pad", [0, 1], ids=["aligned_out", "unaligned_out"])
def test_pair_both_tile_widths(M, N, K, pad):
    """The same product with an Out pitch of N (rows 32-byte aligned: 256-wide
    tiles, one accumulator, epilogue from registers) and N + 1 (192-wide
    tiles, two accumulators, staged epilogue); columns past N untouched."""
    import torch
    A, SA, B, SB = draw(1, M, N, K, "e4m3", seed=M + K)
    ref, absdot = oracle.gemm_nt_mx(A, SA, B, SB, dtype="e4m3")
    a, pa = gpu_util.to_device(A, "e4m3", K)
    b, pb = gpu_util.to_device(B, "e4m3")
    sa = gnt.pack_mx_scales(torch.from_numpy(SA).cuda(), K)
    sb = gnt.pack_mx_scales(torch.from_numpy(SB).cuda(), K)
    ldo = N + pad
    o = torch.full((M, ldo), float("nan"), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    gnt.gemm_nt_mx(pa, sa.data_ptr(), pb, sb.data_ptr(), o.data_ptr(), gnt.DType.E4M3, gnt.DType.F32, M, N, K,
                   K, K, ldo, 0, 0, 0, 1, P.TC05_PAIR, stream)
    gnt.gemm_nt_check(stream)
    got = o.double().cpu().numpy()
    if pad:
        assert np.isnan(got[:, N:]).all()
    check_tol(got[None, :, :N], ref, absdot, "f32", "pair ldo=%d" % ldo)
