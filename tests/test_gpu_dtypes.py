"""bfloat16 inputs and float16 / bfloat16 outputs (gemm_nt_batched_ex) on every
kernel, against the oracle.

"Warp Matrix Instructions", "Other Fragment Shapes and Transfers", names the
bfloat16 form of the same product beside the float16 one; the accumulator stays
float32 in both.  A 16-bit Out is that float32 accumulator rounded once to
nearest even, so the tolerance adds half a unit in the last place of the output
format, and with integer inputs (exact float32 sums) Out must equal the oracle's
rounding of the exact result bit for bit.
"""
import numpy as np
import pytest

import dense_fp16_tensor_gemm_gb300 as gnt
import gpu_util
import oracle
import workloads

pytestmark = pytest.mark.gpu

P = gnt.Path
AB = ["f16", "bf16"]
OUT = ["f32", "f16", "bf16"]


_torch_dtype = gpu_util.torch_dtype
_code = gpu_util.dtype_code
_to_device = gpu_util.to_device
check = gpu_util.check_tol
check_exact = gpu_util.check_exact


def _inputs(batch, M, N, K, ab, dist="normal", seed=0):
    return workloads.make_inputs(batch, M, N, K, dist, 1.0, seed=seed, dtype=ab)


def run_ex(A, B, ab, out, path, ldo=None, out_offset=0, lda=None, ldb=None):
    """Out = A @ B.T through gemm_nt_batched_ex (K-major operands); Out as
    float64 numpy (batch, M, N), nothing written outside it."""
    import torch
    batch, M, K = A.shape
    N = B.shape[1]
    ldo = ldo or N
    lda = lda or K
    ldb = ldb or K
    a, pa = _to_device(A, ab, lda)
    b, pb = _to_device(B, ab, ldb)
    o = torch.full((out_offset + batch * M * ldo,), float("nan"), dtype=_torch_dtype(out), device="cuda")
    esize = o.element_size()
    stream = torch.cuda.current_stream().cuda_stream
    gnt.gemm_nt_batched_ex(pa, pb, o.data_ptr() + esize * out_offset, _code(ab), _code(out), M, N, K,
                           lda, ldb, ldo, M * lda, N * ldb, M * ldo, batch, path, stream)
    gnt.gemm_nt_check(stream)
    host = o.double().cpu().numpy()
    assert np.all(np.isnan(host[:out_offset])), "kernel wrote before the Out base"
    host = host[out_offset:].reshape(batch, M, ldo)
    if ldo > N:
        assert np.all(np.isnan(host[:, :, N:])), "kernel wrote past column N"
    return host[:, :, :N]


@pytest.mark.parametrize("out", OUT)
@pytest.mark.parametrize("ab", AB)
@pytest.mark.parametrize("path", [P.AUTO, P.TC05, P.TC05_PAIR, P.MMASYNC])
def test_ragged_batched(path, ab, out):
    """Several tiles in each direction, ragged M/N/K tails, batch 2."""
    A, B = _inputs(2, 300, 520, 264, ab, seed=101)
    ref, absdot = oracle.gemm_nt(A, B, dtype=ab)
    check(run_ex(A, B, ab, out, path), ref, absdot, out, "%s %s->%s" % (path.name, ab, out))


@pytest.mark.parametrize("out", OUT)
@pytest.mark.parametrize("ab", AB)
@pytest.mark.parametrize("path", [P.TC05, P.TC05_PAIR, P.SKINNY, P.MMASYNC])
def test_integer_inputs_round_exactly(path, ab, out):
    """Integer inputs in [-4,4] with K = 1000: the float32 accumulator is the
    exact integer (up to 16000), so Out is its correctly rounded value; float16
    outputs above 2048 exercise ties and inexact rounding."""
    M = 48 if path == P.SKINNY else 200
    A, B = _inputs(1, M, 1100, 1000, ab, dist="int4", seed=102)
    ref, _ = oracle.gemm_nt(A, B, dtype=ab)
    check_exact(run_ex(A, B, ab, out, path), ref, out, "%s %s->%s" % (path.name, ab, out))


@pytest.mark.parametrize("out", OUT)
@pytest.mark.parametrize("ab", AB)
@pytest.mark.parametrize("M,N,K", [(1, 1024, 64), (33, 1500, 1000), (64, 4096, 520)])
def test_skinny(M, N, K, ab, out):
    A, B = _inputs(1, M, N, K, ab, seed=M + N)
    ref, absdot = oracle.gemm_nt(A, B, dtype=ab)
    check(run_ex(A, B, ab, out, P.SKINNY), ref, absdot, out, "SKINNY %s->%s" % (ab, out))


@pytest.mark.parametrize("out", ["f16", "bf16"])
@pytest.mark.parametrize("path,ldo,out_offset", [
    (P.TC05_PAIR, 520, 0),   # aligned Out rows: direct TMEM -> global epilogue
    (P.TC05_PAIR, 523, 0),   # odd pitch: staged epilogue
    (P.TC05_PAIR, 520, 3),   # base off by 3 elements: staged epilogue
    (P.TC05, 520, 0),        # 4-wide stores
    (P.TC05, 522, 1),        # scalar stores
])
def test_out_layouts(path, ldo, out_offset, out):
    """16-bit Out with padded and offset rows selects each store variant."""
    A, B = _inputs(1, 390, 520, 200, "bf16", seed=103)
    ref, absdot = oracle.gemm_nt(A, B, dtype="bf16")
    got = run_ex(A, B, "bf16", out, path, ldo=ldo, out_offset=out_offset)
    check(got, ref, absdot, out, "%s ldo=%d off=%d ->%s" % (path.name, ldo, out_offset, out))


@pytest.mark.parametrize("ab", AB)
def test_padded_and_misaligned_inputs(ab):
    """Padded leading dimensions (TMA maps with a row pitch) and an input base
    that is not 16-byte aligned (the warp kernel) on bfloat16 / float16."""
    A, B = _inputs(1, 150, 140, 136, ab, seed=104)
    ref, absdot = oracle.gemm_nt(A, B, dtype=ab)
    check(run_ex(A, B, ab, "f32", P.AUTO, lda=200, ldb=144), ref, absdot, "f32", "padded")
    import torch
    a, pa = _to_device(A, ab, offset=1)
    b, pb = _to_device(B, ab)
    o = torch.full((150, 140), float("nan"), dtype=torch.float16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert gnt.gemm_nt_select_path(pa, pb, o.data_ptr(), 150, 140, 136, 136, 136, 140) == P.MMASYNC
    gnt.gemm_nt_batched_ex(pa, pb, o.data_ptr(), _code(ab), gnt.DType.F16, 150, 140, 136, 136, 136, 140,
                           0, 0, 0, 1, P.AUTO, stream)
    gnt.gemm_nt_check(stream)
    check(o.double().cpu().numpy()[None], ref, absdot, "f16", "misaligned")


@pytest.mark.parametrize("out", ["f16", "bf16"])
def test_long_k_few_tiles_with_16_bit_out(out):
    """Few tiles and a long K, where a float32 Out would be split across CTA
    pairs; 16-bit outputs take whole tiles and must still match."""
    A, B = _inputs(1, 512, 512, 8192, "bf16", seed=105)
    ref, absdot = oracle.gemm_nt(A, B, dtype="bf16")
    for path in (P.AUTO, P.TC05_PAIR, P.TC05):
        check(run_ex(A, B, "bf16", out, path), ref, absdot, out, "%s ->%s" % (path.name, out))


def test_torch_wrappers():
    import torch
    A, B = _inputs(3, 130, 250, 192, "bf16", seed=106)
    ref, absdot = oracle.gemm_nt(A, B, dtype="bf16")
    a = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16).cuda()
    b = torch.from_numpy(B.view(np.int16)).view(torch.bfloat16).cuda()
    out = gnt.gemm_nt_batched(a, b, out_dtype=torch.bfloat16)
    assert out.dtype == torch.bfloat16 and tuple(out.shape) == (3, 130, 250)
    check(out.double().cpu().numpy(), ref, absdot, "bf16", "batched wrapper")
    out2 = gnt.gemm_nt(a[1], b[1])
    assert out2.dtype == torch.float32
    check(out2.double().cpu().numpy()[None], ref[1:2], absdot[1:2], "f32", "2-D wrapper")
    out3 = torch.empty((130, 250), dtype=torch.float16, device="cuda")
    gnt.gemm_nt(a[2], b[2], out=out3)
    check(out3.double().cpu().numpy()[None], ref[2:3], absdot[2:3], "f16", "given out")
    with pytest.raises(TypeError):
        gnt.gemm_nt(a[0], b[0].half())
    torch.cuda.synchronize()


def test_bf16_square_4096_sampled():
    """The square 4096 workload's recipe (uniform[-1,1], seed 1) in bfloat16,
    bfloat16 Out, checked on sampled rows, columns and random elements."""
    import gpu_util
    w = workloads.WORKLOADS["square_4096"]
    A, B = workloads.make_inputs(1, w.M, w.N, w.K, w.dist, w.sigma, w.seed, dtype="bf16")
    got = run_ex(A, B, "bf16", "bf16", P.AUTO)
    bb, ii, jj = gpu_util.sample_indices(1, w.M, w.N, 4000, rows=(0, 127, 128, -1), cols=(0, 255, -1))
    ref, absdot = oracle.gemm_nt_sampled(A, B, bb, ii, jj, dtype="bf16")
    check(got[bb, ii, jj], ref, absdot, "bf16", "square_4096 bf16")


@pytest.mark.parametrize("out", ["f16", "bf16"])
def test_k_zero_writes_zeros(out):
    import torch
    o = torch.full((2, 70, 90), float("nan"), dtype=_torch_dtype(out), device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    gnt.gemm_nt_batched_ex(16, 16, o.data_ptr(), gnt.DType.BF16, _code(out), 70, 90, 0, 0, 0, 90, 0, 0,
                           70 * 90, 2, P.AUTO, stream)
    gnt.gemm_nt_check(stream)
    assert bool(torch.all(o == 0))
