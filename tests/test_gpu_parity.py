"""GPU parity: every kernel path of libgemm_nt against the CPU oracle on the
same seeded inputs, through the C ABI.

Tolerance (from the product's definition with fp32 accumulation of exact fp16
products): |Out - ref| <= 1e-3 * sum_k |a_ik * b_jk| + 1e-6 per element, and
Out == ref exactly for integer-valued inputs whose partial sums stay below 2**24.
"""
import numpy as np
import pytest

import dense_fp16_tensor_gemm_gb300 as gnt
import oracle
import workloads
from gpu_util import assert_parity, run_path

pytestmark = pytest.mark.gpu

P = gnt.Path

# Small and ragged shapes: several tiles in each dimension plus partial tiles,
# K tails inside a 64-wide k-block and across 16-wide MMA slices.
SHAPES = [
    (128, 64, 64), (1, 1, 8), (3, 5, 16), (16, 8, 16), (127, 129, 72), (129, 127, 64),
    (200, 300, 136), (257, 513, 200), (384, 256, 64 * 9 + 8), (64, 1000, 520), (1000, 64, 64),
    (333, 777, 1000),
]


@pytest.fixture(scope="module", autouse=True)
def built():
    from dense_fp16_tensor_gemm_gb300 import _build
    _build.build()
    gnt.load()


@pytest.mark.parametrize("path", [P.AUTO, P.TC05, P.TC05_PAIR, P.MMASYNC])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_small_shapes(path, M, N, K):
    A, B = workloads.make_inputs(0, M, N, K, "uniform", seed=M * 7 + N * 3 + K)
    ref, absdot = oracle.gemm_nt(A, B)
    out = run_path(A, B, path)
    assert_parity(out, ref, absdot, what="%s %dx%dx%d" % (path.name, M, N, K))


# Swapped-operand shapes covering its three work distributions on a 152-SM
# GB300: whole tiles (few k-blocks), stream-K (few tiles, long K) and the row
# split (64..128 rows of N per CTA: N = 9728 and 19456 are its two ends).
@pytest.mark.parametrize("M,N,K", [(1, 1024, 64), (7, 2000, 136), (64, 4096, 520), (33, 1500, 1000),
                                   (16, 4096, 8192), (64, 16384, 256), (50, 12001, 200),
                                   (3, 19456, 72), (1, 9728, 512), (32, 9728, 264), (33, 19456, 136),
                                   (64, 13000, 1000)])
def test_skinny_shapes(M, N, K):
    A, B = workloads.make_inputs(0, M, N, K, "normal", 0.02, seed=M + N + K)
    ref, absdot = oracle.gemm_nt(A, B)
    out = run_path(A, B, P.SKINNY)
    assert_parity(out, ref, absdot, what="SKINNY %dx%dx%d" % (M, N, K))


@pytest.mark.parametrize("path", [P.TC05, P.TC05_PAIR, P.SKINNY, P.MMASYNC])
def test_integer_inputs_bit_exact(path):
    M = 48 if path == P.SKINNY else 300
    A, B = workloads.make_inputs(0, M, 1100, 1000, "int4", seed=4)
    ref, absdot = oracle.gemm_nt(A, B)
    assert_parity(run_path(A, B, path), ref, absdot, exact=True, what=path.name)


@pytest.mark.parametrize("path", [P.AUTO, P.TC05, P.TC05_PAIR, P.MMASYNC])
def test_padded_leading_dimensions(path):
    A, B = workloads.make_inputs(0, 190, 270, 200, "uniform", seed=5)
    ref, absdot = oracle.gemm_nt(A, B)
    out = run_path(A, B, path, lda=208, ldb=264, ldo=301)
    assert_parity(out, ref, absdot, what=path.name)


# fp32 Out rows off 16-byte boundaries: the epilogue stores whole 128-byte lines,
# rotating each row by its offset into a line.  Odd ldo gives every row its own
# rotation, ldo = 2 (mod 4) two rows per rotation, and ldo = 0 (mod 32) with a
# base one float off the same rotation on every row.  Shapes end inside a warp's
# 32 rows and inside a 32-column chunk; integer inputs make the result exact.
@pytest.mark.parametrize("path", [P.AUTO, P.TC05, P.TC05_PAIR])
@pytest.mark.parametrize("M,N,ldo,o_offset", [(300, 517, 517, 0), (300, 517, 519, 3), (133, 700, 702, 0),
                                              (133, 700, 704, 1), (261, 290, 320, 1), (40, 1000, 1001, 2),
                                              (513, 77, 77, 5)])
def test_misaligned_out_rows(path, M, N, ldo, o_offset):
    A, B = workloads.make_inputs(0, M, N, 264, "int4", seed=M + N)
    ref, absdot = oracle.gemm_nt(A, B)
    out = run_path(A, B, path, ldo=ldo, o_offset=o_offset)
    assert_parity(out, ref, absdot, exact=True, what="%s %dx%d ldo %d offset %d" % (path.name, M, N, ldo, o_offset))


def test_misaligned_inputs_use_warp_kernel():
    A, B = workloads.make_inputs(0, 100, 90, 77, "uniform", seed=6)
    ref, absdot = oracle.gemm_nt(A, B)
    # odd K (row pitch not a multiple of 16 bytes) and a base off by one element
    assert_parity(run_path(A, B, P.AUTO, a_offset=1), ref, absdot, what="AUTO misaligned")
    assert_parity(run_path(A, B, P.MMASYNC, a_offset=1, b_offset=3), ref, absdot, what="MMASYNC")
    with pytest.raises(gnt.GemmError) as e:
        run_path(A, B, P.TC05, a_offset=1)
    assert e.value.status == gnt.Status.NOT_SUPPORTED


@pytest.mark.parametrize("path", [P.AUTO, P.TC05, P.TC05_PAIR, P.MMASYNC])
def test_batched_ragged(path):
    A, B = workloads.make_inputs(3, 301, 207, 104, "int4", seed=4)
    ref, absdot = oracle.gemm_nt(A, B)
    assert_parity(run_path(A, B, path), ref, absdot, exact=True, what="batched " + path.name)


def test_batched_shared_operand():
    """strideB = 0: every batch multiplies by the same B."""
    import torch
    A, B = workloads.make_inputs(4, 140, 150, 128, "uniform", seed=8)
    B0 = B[0]
    ref, absdot = oracle.gemm_nt(A, np.broadcast_to(B0, B.shape).copy())
    a = torch.from_numpy(A).cuda()
    b = torch.from_numpy(B0).cuda().unsqueeze(0).expand(4, -1, -1)
    for path in (P.AUTO, P.TC05_PAIR, P.MMASYNC):
        out = gnt.gemm_nt_batched(a, b, path=path)
        gnt.gemm_nt_check()
        assert_parity(out.cpu().numpy(), ref, absdot, what="shared B " + path.name)


def test_k_zero_and_empty():
    import torch
    out = torch.full((5, 7), 3.0, device="cuda")
    a = torch.empty((5, 0), dtype=torch.float16, device="cuda")
    b = torch.empty((7, 0), dtype=torch.float16, device="cuda")
    gnt.gemm_nt_f16_f32(a.data_ptr(), b.data_ptr(), out.data_ptr(), 5, 7, 0, 0, 0, 7)
    gnt.gemm_nt_check()
    assert torch.all(out == 0)
    gnt.gemm_nt_f16_f32(0, 0, out.data_ptr(), 0, 7, 16, 16, 16, 7)  # M = 0: nothing
    gnt.gemm_nt_check()


def test_torch_wrapper_and_streams():
    import torch
    A, B = workloads.make_inputs(0, 256, 384, 320, "uniform", seed=9)
    ref, absdot = oracle.gemm_nt(A, B)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a, b = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        out = gnt.gemm_nt(a, b)
    s.synchronize()
    gnt.gemm_nt_check(s.cuda_stream)
    assert_parity(out.cpu().numpy(), ref, absdot, what="torch wrapper")


@pytest.mark.parametrize("batch,M,N,K", [(2, 130, 260, 192), (5, 70, 90, 64), (1, 2000, 300, 136),
                                         (1, 100, 50, 40), (1, 2500, 2100, 136), (1, 2048, 2048, 64)])
def test_from_host_pipeline(batch, M, N, K):
    """Host buffers in and out; chunks of batches or of rows, or for a large
    single product 4 x 4 blocks of Out (uneven ones for 2500 x 2100), overlap
    the copies."""
    import torch
    A, B = workloads.make_inputs(batch, M, N, K, "uniform", seed=10)
    ref, absdot = oracle.gemm_nt(A, B)
    ha = torch.from_numpy(A).pin_memory()
    hb = torch.from_numpy(B).pin_memory()
    ho = torch.full((batch, M, N), float("nan"), dtype=torch.float32).pin_memory()
    da = torch.empty_like(ha, device="cuda")
    db = torch.empty_like(hb, device="cuda")
    do = torch.empty_like(ho, device="cuda")
    st = torch.cuda.current_stream()
    for _ in range(2):  # twice: the second call reuses the streams and events
        gnt.gemm_nt_f16_f32_from_host(ha.data_ptr(), hb.data_ptr(), ho.data_ptr(), da.data_ptr(),
                                      db.data_ptr(), do.data_ptr(), M, N, K, batch, st.cuda_stream)
        gnt.gemm_nt_check(st.cuda_stream)
        assert_parity(ho.numpy(), ref, absdot, what="from_host")
        ho.fill_(float("nan"))


def test_coded_inputs_show_row_per_thread_map():
    """"Blackwell Tensor Cores": thread t of the epilogue warpgroup holds
    accumulator row t.  With A[i,0] = i (else 0) and B[j,0] = 1, Out[i,j] = i;
    with A[i,0] = 1 and B[j,0] = j, Out[i,j] = j.  Any lane or column mix-up in
    the TMEM read-out shows as a wrong row or column value."""
    for path, (M, N, K) in ((P.TC05, (128, 64, 64)), (P.TC05_PAIR, (256, 256, 64))):
        A = np.zeros((M, K), np.float16); B = np.zeros((N, K), np.float16)
        A[:, 0] = np.arange(M); B[:, 0] = 1
        out = run_path(A, B, path)
        assert np.array_equal(out, np.repeat(np.arange(M, dtype=np.float32)[:, None], N, 1)), path.name
        A[:, 0] = 1; B[:, 0] = np.arange(N)
        out = run_path(A, B, path)
        assert np.array_equal(out, np.repeat(np.arange(N, dtype=np.float32)[None, :], M, 0)), path.name


def test_identity_and_permutation():
    rng = np.random.default_rng(12)
    K = 256
    A = rng.standard_normal((300, K)).astype(np.float16)
    I = np.eye(K, dtype=np.float16)
    p = rng.permutation(K)
    Pm = np.zeros((K, K), np.float16); Pm[np.arange(K), p] = 1
    for path in (P.TC05, P.TC05_PAIR, P.MMASYNC):
        assert np.array_equal(run_path(A, I, path), A.astype(np.float32))
        assert np.array_equal(run_path(A, Pm, path), A.astype(np.float32)[:, p])


# Shapes that put the CTA-pair kernel in stream-K mode on a 152-SM GB300 (76
# pairs): far fewer tiles than pairs and at least 96 k-blocks, with ragged M/N
# and K tails and batches; (1024, 1024, 4096) stays on whole tiles.
SK_SHAPES = [(512, 512, 8192, 0), (700, 900, 7000, 0), (300, 500, 6504, 3), (1024, 1024, 6144, 0),
             (1024, 1024, 4096, 0)]


@pytest.mark.parametrize("M,N,K,batch", SK_SHAPES)
def test_pair_stream_k(M, N, K, batch):
    A, B = workloads.make_inputs(batch, M, N, K, "uniform", seed=M + N + K)
    ref, absdot = oracle.gemm_nt(A, B)
    assert_parity(run_path(A, B, P.TC05_PAIR), ref, absdot, what="pair stream-K %s" % ((M, N, K, batch),))


def test_pair_stream_k_integer_exact_and_deterministic():
    A, B = workloads.make_inputs(0, 512, 512, 8192, "int4", seed=4)
    ref, absdot = oracle.gemm_nt(A, B)
    out1 = run_path(A, B, P.TC05_PAIR)
    assert_parity(out1, ref, absdot, exact=True, what="pair stream-K integers")
    A, B = workloads.make_inputs(0, 512, 512, 8192, "normal", 1.0, seed=5)
    o1, o2 = run_path(A, B, P.TC05_PAIR), run_path(A, B, P.TC05_PAIR)
    assert np.array_equal(o1.view(np.uint32), o2.view(np.uint32)), "stream-K sum order is not fixed"


@pytest.mark.parametrize("batch,M,N,K", [(2, 600, 1024, 1000), (1, 513, 768, 2000)])
def test_epilogue_choice_keeps_every_bit(batch, M, N, K):
    """The pair kernel stores Out straight from TMEM when A's and B's rows sit on
    128-byte lines, and through shared memory otherwise (rows of K = 1000
    elements are 2000 bytes apart).  Both epilogues store the same accumulator:
    the products must agree bit for bit with each other, and with the oracle."""
    A, B = workloads.make_inputs(batch, M, N, K, "normal", 1.0, seed=batch + M + K)
    ref, absdot = oracle.gemm_nt(A, B)
    pitch = (K + 63) // 64 * 64  # whole 128-byte lines
    packed = run_path(A, B, P.TC05_PAIR)                                  # 2000- / 4000-byte rows
    padded = run_path(A, B, P.TC05_PAIR, lda=pitch, ldb=pitch)           # rows on 128-byte lines
    assert_parity(packed, ref, absdot, what="pair, rows off their lines")
    assert_parity(padded, ref, absdot, what="pair, rows on lines")
    assert np.array_equal(packed, padded)
