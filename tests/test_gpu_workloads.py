"""GPU parity on the five named workloads at full size, in the configuration
bench.py times (automatic path, packed layouts).

The oracle computes sampled elements one by one: random elements plus whole
rows and columns at tile borders and at the ragged ends.  The integer batch is
checked bit-exact on its samples, and on every element through two exact
properties: every output is an integer, and the row and column sums equal
sum_k A[i,k] * (sum_j B[j,k]) and sum_k B[j,k] * (sum_i A[i,k]) in int64.
"""
import numpy as np
import pytest

import dense_fp16_tensor_gemm_gb300 as gnt
import oracle
import workloads
from gpu_util import sample_indices

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from dense_fp16_tensor_gemm_gb300 import _build
    _build.build()
    gnt.load()


def run_auto(A, B):
    import torch
    a, b = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    out = gnt.gemm_nt_batched(a, b) if A.ndim == 3 else gnt.gemm_nt(a, b)
    gnt.gemm_nt_check()
    return out.cpu().numpy()


def check_sampled(A, B, out, rows, cols, n_random, exact=False, seed=0):
    A3 = A[None] if A.ndim == 2 else A
    B3 = B[None] if B.ndim == 2 else B
    o3 = out[None] if out.ndim == 2 else out
    batch, M, _ = A3.shape
    N = B3.shape[1]
    bi, ii, jj = sample_indices(batch, M, N, n_random, rows, cols, seed)
    ref, absdot = oracle.gemm_nt_sampled(A3, B3, bi, ii, jj)
    got = o3[bi, ii, jj].astype(np.float64)
    assert not np.isnan(got).any()
    bad = (got != ref) if exact else ~oracle.within_tolerance(got, ref, absdot)
    assert not bad.any(), "%d of %d sampled elements out of tolerance, e.g. (b,i,j)=%s got %r ref %r" % (
        int(bad.sum()), bad.size, (bi[bad][0], ii[bad][0], jj[bad][0]), got[bad][0], ref[bad][0])


def test_tile_128x64x64_full():
    A, B = workloads.workload_inputs("tile_128x64x64")
    ref, absdot = oracle.gemm_nt(A, B)
    for path in (gnt.Path.AUTO, gnt.Path.TC05, gnt.Path.MMASYNC):
        import torch
        out = gnt.gemm_nt(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), path=path)
        gnt.gemm_nt_check()
        assert oracle.within_tolerance(out.cpu().numpy(), ref, absdot).all(), path.name


def test_square_4096():
    A, B = workloads.workload_inputs("square_4096")
    out = run_auto(A, B)
    check_sampled(A, B, out, rows=(0, 127, 128, -1), cols=(0, 255, 256, -1), n_random=4096)


def test_square_8192():
    A, B = workloads.workload_inputs("square_8192")
    out = run_auto(A, B)
    check_sampled(A, B, out, rows=(0, 128, 4095, -1), cols=(0, 255, 256, -1), n_random=4096)


def test_skinny_64x16384x8192():
    A, B = workloads.workload_inputs("skinny_64x16384x8192")
    out = run_auto(A, B)
    check_sampled(A, B, out, rows=(0, 31, -1), cols=(0, 127, 128, 8191, -1), n_random=4096)


def test_ragged_batch16_exact():
    A, B = workloads.workload_inputs("ragged_batch16_3001x2047x1000")
    out = run_auto(A, B)
    check_sampled(A, B, out, rows=(0, 127, 128, -1), cols=(0, 255, 256, -1), n_random=1024, exact=True)
    o = out.astype(np.float64)
    assert np.array_equal(o, np.round(o)), "non-integer outputs"
    ai, bi = A.astype(np.int64), B.astype(np.int64)
    row_sums = np.einsum("bik,bk->bi", ai, bi.sum(axis=1))
    col_sums = np.einsum("bjk,bk->bj", bi, ai.sum(axis=1))
    assert np.array_equal(o.sum(axis=2), row_sums.astype(np.float64)), "row sums"
    assert np.array_equal(o.sum(axis=1), col_sums.astype(np.float64)), "column sums"
