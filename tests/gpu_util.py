"""Helpers for the GPU tests: move seeded numpy inputs to the device, run one
library path through the C ABI, and compare with the oracle."""
import numpy as np

import dense_fp16_tensor_gemm_gb300 as gnt
import oracle


def dev(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def run_path(A, B, path, lda=None, ldb=None, ldo=None, a_offset=0, b_offset=0, o_offset=0):
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
    # Out's elements before the (offset) base and past column N hold NaN and must stay so
    flat = torch.full((o_offset + batch * M * ldo,), float("nan"), dtype=torch.float32, device="cuda")
    gnt.gemm_nt_f16_f32_batched_path(
        a.data_ptr() + 2 * a_offset, b.data_ptr() + 2 * b_offset, flat.data_ptr() + 4 * o_offset, M, N, K, lda,
        ldb, ldo, M * lda, N * ldb, M * ldo, batch, path, torch.cuda.current_stream().cuda_stream)
    gnt.gemm_nt_check(torch.cuda.current_stream().cuda_stream)
    f = flat.cpu().numpy()
    assert np.all(np.isnan(f[:o_offset])), "kernel wrote before Out's base"
    o = f[o_offset:].reshape(batch, M, ldo)
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


TORCH_DTYPES = ("f16", "bf16", "f32")


def torch_dtype(name):
    import torch
    return {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32,
            "e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2,
            "e2m3": torch.uint8, "e3m2": torch.uint8, "e2m1": torch.uint8}[name]


def dtype_code(name):
    return {"f16": gnt.DType.F16, "bf16": gnt.DType.BF16, "f32": gnt.DType.F32,
            "e4m3": gnt.DType.E4M3, "e5m2": gnt.DType.E5M2, "e2m3": gnt.DType.E2M3, "e3m2": gnt.DType.E3M2,
            "e2m1": gnt.DType.E2M1}[name]


def esize(name):
    return {"f16": 2, "bf16": 2, "f32": 4, "e4m3": 1, "e5m2": 1, "e2m3": 1, "e3m2": 1, "e2m1": 1}[name]


def to_device(bits, ab, ld=None, offset=0):
    """(batch, rows, cols) host array of bit patterns (float16 or uint16 for
    the 16-bit types, uint8 for the 8-bit floats) -> device tensor of dtype
    `ab` with row pitch `ld`; padding and the `offset` elements before the base
    hold NaN.  Returns (tensor, base pointer)."""
    import torch
    es = esize(ab)
    x = np.ascontiguousarray(bits).view(np.int16 if es == 2 else np.uint8)
    batch, rows, cols = x.shape
    ld = ld or cols
    t = torch.full((offset + batch * rows * ld,), float("nan"), dtype=torch.float32).to(torch_dtype(ab))
    t[offset:].view(batch, rows, ld)[:, :, :cols] = torch.from_numpy(x.copy()).view(torch_dtype(ab))
    t = t.cuda()
    return t, t.data_ptr() + es * offset


PACKED = {"e2m3": 6, "e3m2": 6, "e2m1": 4}  # bits per element of the packed types


def to_device_packed(codes, ab, ld):
    """(batch, rows, K) codes of a packed 6- or 4-bit type -> device bytes in
    the packed storage with a row pitch of `ld` elements (padding zero).
    Returns (tensor, base pointer)."""
    import torch
    import workloads
    bits = PACKED[ab]
    batch, rows, K = codes.shape
    packed = workloads.pack_subbyte(codes, ab)
    pitch = ld * bits // 8
    t = torch.zeros(batch * rows * pitch, dtype=torch.uint8)
    t.view(batch, rows, pitch)[:, :, :packed.shape[2]] = torch.from_numpy(packed)
    t = t.cuda()
    return t, t.data_ptr()


def run_general(A, B, ab, out, path, a_mn=False, b_mn=False, lda=None, ldb=None, ldo=None, out_offset=0,
                a_offset=0):
    """Out = A @ B.T through gemm_nt_batched_major, A (batch, M, K) and B
    (batch, N, K) the logical operands; an MN-major operand is handed to the
    library as its transpose (batch, K, rows), row pitch lda / ldb (default:
    the stored row length, rounded up to 8 for an MN-major operand).  Returns Out
    as float64 numpy (batch, M, N) after checking that nothing beyond column N
    or before the Out base was written."""
    import torch
    batch, M, K = A.shape
    N = B.shape[1]
    As = np.ascontiguousarray(np.swapaxes(A, 1, 2)) if a_mn else A
    Bs = np.ascontiguousarray(np.swapaxes(B, 1, 2)) if b_mn else B
    # default pitch of an MN-major operand: its row length (M or N) rounded up
    # to 8 elements, the alignment the tensor-core kernels need
    lda = lda or ((As.shape[2] + 7) // 8 * 8 if a_mn else As.shape[2])
    ldb = ldb or ((Bs.shape[2] + 7) // 8 * 8 if b_mn else Bs.shape[2])
    ldo = ldo or N
    if ab in PACKED:
        a, pa = to_device_packed(As, ab, lda)
        b, pb = to_device_packed(Bs, ab, ldb)
    else:
        a, pa = to_device(As, ab, lda, a_offset)
        b, pb = to_device(Bs, ab, ldb)
    o = torch.full((out_offset + batch * M * ldo,), float("nan"), dtype=torch_dtype(out), device="cuda")
    esize = o.element_size()
    stream = torch.cuda.current_stream().cuda_stream
    gnt.gemm_nt_batched_major(pa, gnt.Major.MN if a_mn else gnt.Major.K, pb, gnt.Major.MN if b_mn else gnt.Major.K,
                              o.data_ptr() + esize * out_offset, dtype_code(ab), dtype_code(out), M, N, K,
                              lda, ldb, ldo, As.shape[1] * lda, Bs.shape[1] * ldb, M * ldo, batch, path, stream)
    gnt.gemm_nt_check(stream)
    host = o.double().cpu().numpy()
    assert np.all(np.isnan(host[:out_offset])), "kernel wrote before the Out base"
    host = host[out_offset:].reshape(batch, M, ldo)
    if ldo > N:
        assert np.all(np.isnan(host[:, :, N:])), "kernel wrote past column N"
    return host[:, :, :N]


def check_tol(out, ref, absdot, out_dtype, what):
    """Elementwise parity within oracle.within_tolerance for Out's type."""
    assert not np.isnan(out).any(), "%s: unwritten elements" % what
    ok = oracle.within_tolerance(out, ref, absdot, out_dtype)
    if not ok.all():
        i = tuple(np.argwhere(~ok)[0])
        raise AssertionError("%s: %d of %d out of tolerance; first %s out=%r ref=%r absdot=%r"
                             % (what, int((~ok).sum()), ok.size, i, out[i], ref[i], absdot[i]))


def check_exact(out, ref, out_dtype, what):
    """Out equals the oracle's rounding of an exact result into Out's type."""
    want = oracle.round_output(ref, out_dtype)
    bad = out != want
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError("%s: %d of %d differ from the rounded exact result; first %s out=%r want=%r"
                             % (what, int(bad.sum()), bad.size, i, out[i], want[i]))
