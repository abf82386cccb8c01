"""Helpers for the GPU tests: move seeded numpy inputs to the device, run one
library path through the C ABI, and compare with the oracle."""
import numpy as np

import dense_fp16_tensor_gemm_gb300 as gnt
import oracle


def dev(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def run_path(A, B, path, lda=None, ldb=None, ldo=None, a_offset=0, b_offset=0):
    """Out = A @ B.T through gemm_nt_f16_f32_batched_path.

    A (M,K) or (batch,M,K), B likewise, numpy float16.  Optional padded leading
    dimensions and element offsets of the device bases (to make them
    misaligned) exercise the layout handling.  Returns numpy float32 Out.
    """
    import torch
    A3 = A[None] if A.ndim == 2 else A
    B3 = B[None] if B.ndim == 2 else B
    batch, M, K = A3.shape
    N = B3.shape[1]
    lda = lda or K
    ldb = ldb or K
    ldo = ldo or N
    # padding (beyond K, before the offset base) holds NaN: reading it poisons Out
    a = torch.full((a_offset + batch * M * lda,), float("nan"), dtype=torch.float16)
    a[a_offset:].view(batch, M, lda)[:, :, :K] = torch.from_numpy(A3)
    b = torch.full((b_offset + batch * N * ldb,), float("nan"), dtype=torch.float16)
    b[b_offset:].view(batch, N, ldb)[:, :, :K] = torch.from_numpy(B3)
    a, b = a.cuda(), b.cuda()
    out = torch.full((batch, M, ldo), float("nan"), dtype=torch.float32, device="cuda")
    gnt.gemm_nt_f16_f32_batched_path(
        a.data_ptr() + 2 * a_offset, b.data_ptr() + 2 * b_offset, out.data_ptr(), M, N, K, lda,
        ldb, ldo, batch, M * lda, N * ldb, M * ldo, path, torch.cuda.current_stream().cuda_stream)
    gnt.gemm_nt_check(torch.cuda.current_stream().cuda_stream)
    o = out.cpu().numpy()
    if ldo > N:
        assert np.all(np.isnan(o[:, :, N:])), "kernel wrote past column N"
    o = o[:, :, :N]
    return o[0] if A.ndim == 2 else o


def assert_parity(out, ref, absdot, exact=False, what=""):
    """|out - ref| <= 1e-3*absdot + 1e-6 elementwise; bit-exact if `exact`."""
    out = np.asarray(out, dtype=np.float64)
    assert out.shape == ref.shape, (out.shape, ref.shape)
    assert not np.isnan(out).any(), "%s: NaN in output (unwritten elements?)" % what
    if exact:
        bad = out != ref
    else:
        bad = ~oracle.within_tolerance(out, ref, absdot)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        details = ["%s: out=%r ref=%r absdot=%r" % (tuple(i), out[tuple(i)], ref[tuple(i)],
                                                     absdot[tuple(i)]) for i in idx]
        raise AssertionError("%s: %d of %d elements out of tolerance; first: %s"
                             % (what, int(bad.sum()), bad.size, "; ".join(details)))


def sample_indices(batch, M, N, n_random, rows=(), cols=(), seed=0):
    """Sample (b, i, j): n_random random elements per batch, plus whole rows and
    whole columns given by index (negative = from the end), in every batch."""
    rng = np.random.default_rng(seed)
    bs, is_, js = [], [], []
    for b in range(batch):
        bs.append(np.full(n_random, b))
        is_.append(rng.integers(0, M, n_random))
        js.append(rng.integers(0, N, n_random))
        for r in rows:
            r = r % M
            bs.append(np.full(N, b)); is_.append(np.full(N, r)); js.append(np.arange(N))
        for c in cols:
            c = c % N
            bs.append(np.full(M, b)); is_.append(np.arange(M)); js.append(np.full(M, c))
    return np.concatenate(bs), np.concatenate(is_), np.concatenate(js)
