"""Pins of the CPU oracle: checks of ``oracle.Oracle`` against facts fixed by
the pages and by mathematics, never against the oracle itself.

Each ``pin_*`` raises AssertionError when the oracle is wrong.  They are run on
the real oracle (tests/test_oracle.py, must pass) and on copies with a planted
mistake (tests/test_oracle_mutants.py, some pin must fail).

Sources:
  * "Warp Matrix Instructions" (opening paragraph and the closing check of
    "From Shared Memory to a Matrix Product"): Out = A @ B.T for A (16,16),
    B (8,16) fp16 with fp32 accumulation, checked with rtol = atol = 2e-4
    against the fp32 product of randn inputs.
  * "Blackwell Tensor Cores", "The Accumulator's Lifetime": the same product
    for A (128,64), B (64,64), same check.
  * "Warp Matrix Instructions", "Other Fragment Shapes and Transfers": the
    same product with bfloat16 inputs.
  * IEEE 754 binary16 (the fp16 format), bfloat16 (the upper 16 bits of an
    IEEE binary32), the 8-bit floats E4M3 and E5M2, and exact rational
    arithmetic.
"""
from fractions import Fraction

import numpy as np

U = 2.0 ** -53  # unit roundoff of IEEE double


def gamma(n):
    """Standard bound factor n*u/(1-n*u) for n sequential double additions."""
    return n * U / (1.0 - n * U)


def exact_product(A16, B16):
    """Exact Out = A @ B.T as (Fraction matrix, exact sum |a*b| matrix).

    Every finite fp16 value is an integer multiple of 2**-24, so scaling by
    2**24 gives integers (computed through float64, which holds them exactly);
    the products and their sums are then exact Python integers (object arrays),
    with value S / 2**48.
    """
    a = (np.asarray(A16, dtype=np.float16).astype(np.float64) * 2.0 ** 24)
    b = (np.asarray(B16, dtype=np.float16).astype(np.float64) * 2.0 ** 24)
    ai = np.vectorize(int, otypes=[object])(a)
    bi = np.vectorize(int, otypes=[object])(b)
    s = ai.dot(bi.T)
    sabs = np.abs(ai).dot(np.abs(bi).T)
    scale = 2 ** 48
    to_frac = np.vectorize(lambda v: Fraction(v, scale), otypes=[object])
    return to_frac(s), to_frac(sabs)


def check_against_exact(orc, A16, B16):
    ref, absdot = orc.gemm_nt(A16, B16)
    exact, exact_abs = exact_product(A16, B16)
    K = np.shape(A16)[-1]
    g = gamma(max(K - 1, 0))
    ex = np.vectorize(float, otypes=[np.float64])(exact)
    exa = np.vectorize(float, otypes=[np.float64])(exact_abs)
    # ref within the summation bound of the exact value; absdot likewise.
    err = np.abs(ref - ex)
    assert np.all(err <= g * exa * (1 + 2 * U) + 2 * U * np.abs(ex) + 1e-300), \
        "oracle differs from the exact sum by more than the double summation bound"
    assert np.all(np.abs(absdot - exa) <= (g + 2 * U) * exa + 1e-300), \
        "absdot differs from the exact sum of |a*b|"
    return ref, absdot, ex


def pin_decoder_exhaustive(orc):
    """All 65536 fp16 bit patterns decode to numpy's float16 -> float64 value."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = orc.half_to_double(bits)
    want = bits.view(np.float16).astype(np.float64)
    nan_g, nan_w = np.isnan(got), np.isnan(want)
    assert np.array_equal(nan_g, nan_w), "NaN patterns decode differently"
    assert np.array_equal(got[~nan_g], want[~nan_w]), "fp16 decoder mismatch"
    # signed zero keeps its sign
    assert np.array_equal(np.signbit(got[~nan_g]), np.signbit(want[~nan_w]))


def pin_bruteforce_tiny(orc, seed=11):
    """Random tiny shapes, including subnormals and extreme fp16 values, equal
    the exact rational sum within the double summation bound."""
    rng = np.random.default_rng(seed)
    specials = np.array([0.0, -0.0, 2.0 ** -24, -(2.0 ** -24), 2.0 ** -14, 65504.0,
                         -65504.0, 1.0, -1.0, 0.5, 3.0], dtype=np.float16)
    for trial in range(40):
        M, N, K = (int(x) for x in rng.integers(1, 9, size=3))
        A = (rng.standard_normal((M, K)) * 4).astype(np.float16)
        B = (rng.standard_normal((N, K)) * 4).astype(np.float16)
        if trial % 3 == 0:
            A.flat[rng.integers(0, A.size, size=min(3, A.size))] = rng.choice(specials, size=min(3, A.size))
            B.flat[rng.integers(0, B.size, size=min(3, B.size))] = rng.choice(specials[:5], size=min(3, B.size))
        check_against_exact(orc, A, B)


def pin_k1_exact(orc):
    """K = 1: a single product of two fp16 values is exact in double."""
    rng = np.random.default_rng(5)
    A = (rng.standard_normal((7, 1)) * 100).astype(np.float16)
    B = (rng.standard_normal((5, 1)) * 0.01).astype(np.float16)
    ref, absdot = orc.gemm_nt(A, B)
    want = A.astype(np.float64) @ B.astype(np.float64).T
    assert np.array_equal(ref, want)
    assert np.array_equal(absdot, np.abs(want))


def pin_worked_examples(orc, seed=3):
    """The two worked-example shapes: exact-sum bound, and the pages' own
    assert_close(rtol=2e-4, atol=2e-4) against the fp32 product."""
    rng = np.random.default_rng(seed)
    for (M, N, K) in ((16, 8, 16), (128, 64, 64)):
        A = rng.standard_normal((M, K)).astype(np.float16)
        B = rng.standard_normal((N, K)).astype(np.float16)
        ref, _, _ = check_against_exact(orc, A, B)
        f32 = A.astype(np.float32) @ B.astype(np.float32).T
        assert np.all(np.abs(ref - f32) <= 2e-4 + 2e-4 * np.abs(f32)), \
            "oracle fails the pages' own fp32 check"


def pin_closed_forms(orc):
    """Products with a known closed form, exactly."""
    # ones: every entry is K
    for K in (1, 7, 64, 1000):
        ref, absdot = orc.gemm_nt(np.ones((3, K), np.float16), np.ones((4, K), np.float16))
        assert np.all(ref == K) and np.all(absdot == K)
    rng = np.random.default_rng(7)
    # identity: B = I_K gives Out = A (each entry is one exact product)
    K = 24
    A = rng.standard_normal((10, K)).astype(np.float16)
    ref, _ = orc.gemm_nt(A, np.eye(K, dtype=np.float16))
    assert np.array_equal(ref, A.astype(np.float64)), "identity product"
    # permutation: B = P gives the columns of A permuted: Out[i,j] = A[i, p[j]]
    p = rng.permutation(K)
    P = np.zeros((K, K), np.float16)
    P[np.arange(K), p] = 1
    ref, _ = orc.gemm_nt(A, P)
    assert np.array_equal(ref, A.astype(np.float64)[:, p]), "permutation product"
    # identity on the left: A = I gives Out = B.T
    B = rng.standard_normal((9, K)).astype(np.float16)
    ref, _ = orc.gemm_nt(np.eye(K, dtype=np.float16), B)
    assert np.array_equal(ref, B.astype(np.float64).T), "left identity"
    # rank one: A[i,k] = x_i, B[j,k] = y_j gives K * x_i * y_j (small integers: exact)
    x = rng.integers(-8, 9, size=6).astype(np.float16)
    y = rng.integers(-8, 9, size=5).astype(np.float16)
    K = 50
    ref, absdot = orc.gemm_nt(np.repeat(x[:, None], K, 1), np.repeat(y[:, None], K, 1))
    want = K * np.outer(x.astype(np.float64), y.astype(np.float64))
    assert np.array_equal(ref, want) and np.array_equal(absdot, np.abs(want))
    # a single nonzero column pair: only k = 3 contributes
    A = np.zeros((4, 8), np.float16)
    B = np.zeros((5, 8), np.float16)
    A[:, 3] = np.arange(1, 5)
    B[:, 3] = -np.arange(1, 6)
    ref, _ = orc.gemm_nt(A, B)
    assert np.array_equal(ref, -np.outer(np.arange(1, 5), np.arange(1, 6)).astype(np.float64))
    # empty sum: K = 0 gives zeros
    ref, absdot = orc.gemm_nt(np.zeros((3, 0), np.float16), np.zeros((2, 0), np.float16))
    assert ref.shape == (3, 2) and np.all(ref == 0) and np.all(absdot == 0)


def pin_integer_exact(orc, seed=4):
    """Integer inputs in [-4,4]: every partial sum is an integer below 2**53,
    so the oracle is exact; compare with integer arithmetic."""
    rng = np.random.default_rng(seed)
    A = rng.integers(-4, 5, size=(2, 37, 300)).astype(np.float16)
    B = rng.integers(-4, 5, size=(2, 29, 300)).astype(np.float16)
    ref, absdot = orc.gemm_nt(A, B)
    ai, bi = A.astype(np.int64), B.astype(np.int64)
    want = np.einsum("bik,bjk->bij", ai, bi)
    wabs = np.einsum("bik,bjk->bij", np.abs(ai), np.abs(bi))
    assert np.array_equal(ref, want.astype(np.float64)), "integer product not exact"
    assert np.array_equal(absdot, wabs.astype(np.float64))


def pin_numpy_crosscheck(orc, seed=9):
    """Mid-size shapes against numpy's float64 matmul (independent code, other
    summation order): both are within gamma_K * absdot of the exact value."""
    rng = np.random.default_rng(seed)
    for (M, N, K) in ((96, 80, 200), (33, 130, 513)):
        A = rng.standard_normal((M, K)).astype(np.float16)
        B = rng.standard_normal((N, K)).astype(np.float16)
        ref, absdot = orc.gemm_nt(A, B)
        want = A.astype(np.float64) @ B.astype(np.float64).T
        assert np.all(np.abs(ref - want) <= 2 * gamma(K) * absdot + 1e-300)
        wabs = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64)).T
        assert np.all(np.abs(absdot - wabs) <= 2 * gamma(K) * wabs + 1e-300)


def pin_batched_and_sampled(orc, seed=13):
    """Batched layout: batch b of the result is the product of batch b of the
    inputs (checked with numpy); sampled elements equal the numpy values."""
    rng = np.random.default_rng(seed)
    batch, M, N, K = 3, 11, 6, 19
    A = rng.integers(-4, 5, size=(batch, M, K)).astype(np.float16)
    B = rng.integers(-4, 5, size=(batch, N, K)).astype(np.float16)
    ref, _ = orc.gemm_nt(A, B)
    want = np.einsum("bik,bjk->bij", A.astype(np.int64), B.astype(np.int64)).astype(np.float64)
    assert np.array_equal(ref, want), "batched product"
    bb = rng.integers(0, batch, size=50)
    ii = rng.integers(0, M, size=50)
    jj = rng.integers(0, N, size=50)
    sref, sabs = orc.gemm_nt_sampled(A, B, bb, ii, jj)
    assert np.array_equal(sref, want[bb, ii, jj]), "sampled product"
    wabs = np.einsum("bik,bjk->bij", np.abs(A.astype(np.int64)), np.abs(B.astype(np.int64)))
    assert np.array_equal(sabs, wabs[bb, ii, jj].astype(np.float64))


def bf16_values(bits):
    """bfloat16 bit patterns -> float64 through the format's definition: the
    pattern is the upper half of an IEEE binary32 whose lower half is zero."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def bf16_bits(x):
    """float64 values that bfloat16 holds exactly -> their bit patterns."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32)
    assert np.all(u & 0xFFFF == 0), "value is not a bfloat16"
    return (u >> 16).astype(np.uint16)


def pin_bf16_decoder_exhaustive(orc):
    """All 65536 bfloat16 bit patterns decode to the binary32 they head."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = orc.bf16_to_double(bits)
    want = bf16_values(bits)
    nan_g, nan_w = np.isnan(got), np.isnan(want)
    assert np.array_equal(nan_g, nan_w), "NaN patterns decode differently"
    assert np.array_equal(got[~nan_g], want[~nan_w]), "bf16 decoder mismatch"
    assert np.array_equal(np.signbit(got[~nan_g]), np.signbit(want[~nan_w]))


def pin_bf16_exact_tiny(orc, seed=21):
    """bfloat16 products over random tiny shapes, with subnormals and values
    near the format's extremes, equal the exact rational sum within the double
    summation bound; batched and sampled elements agree with the full product."""
    rng = np.random.default_rng(seed)
    specials = np.array([0.0, -0.0, 2.0 ** -133, -(2.0 ** -126), 2.0 ** -127 * 3, 1.0, -1.5,
                         2.0 ** 100 * 1.9921875, 255.0, -(2.0 ** -60)])
    for (batch, M, N, K) in ((1, 3, 4, 9), (2, 5, 3, 17), (1, 1, 1, 1), (2, 4, 2, 33)):
        vals_a = rng.choice(specials, size=(batch, M, K))
        vals_b = rng.choice(specials, size=(batch, N, K))
        mix_a = rng.random((batch, M, K)) < 0.5
        mix_b = rng.random((batch, N, K)) < 0.5
        # random normals truncated to bfloat16 (clear the low 16 bits of the binary32)
        na = (rng.standard_normal((batch, M, K)).astype(np.float32).view(np.uint32) & 0xFFFF0000)
        nb = (rng.standard_normal((batch, N, K)).astype(np.float32).view(np.uint32) & 0xFFFF0000)
        a = np.where(mix_a, vals_a, na.view(np.float32).astype(np.float64))
        b = np.where(mix_b, vals_b, nb.view(np.float32).astype(np.float64))
        A, B = bf16_bits(a), bf16_bits(b)
        ref, absdot = orc.gemm_nt(A, B, dtype="bf16")
        assert np.all(np.isfinite(ref)) and np.all(np.isfinite(absdot)), "exact sums here are finite"
        av, bv = bf16_values(A), bf16_values(B)
        g = gamma(max(K - 1, 0))
        for bi in range(batch):
            for i in range(M):
                for j in range(N):
                    terms = [Fraction(float(av[bi, i, k])) * Fraction(float(bv[bi, j, k])) for k in range(K)]
                    ex = sum(terms, Fraction(0))
                    exa = sum((abs(t) for t in terms), Fraction(0))
                    err = abs(Fraction(float(ref[bi, i, j])) - ex)
                    assert err <= Fraction(g) * exa * Fraction(1 + 2 * U) + Fraction(2 * U) * abs(ex) \
                        + Fraction(1, 2 ** 1074), "bf16 product differs from the exact sum"
                    assert abs(Fraction(float(absdot[bi, i, j])) - exa) <= Fraction(g + 2 * U) * exa \
                        + Fraction(1, 2 ** 1074), "bf16 absdot differs from the exact sum"
        bb = rng.integers(0, batch, size=20)
        ii = rng.integers(0, M, size=20)
        jj = rng.integers(0, N, size=20)
        sref, sabs = orc.gemm_nt_sampled(A, B, bb, ii, jj, dtype="bf16")
        assert np.array_equal(sref, ref[bb, ii, jj]) and np.array_equal(sabs, absdot[bb, ii, jj])


def pin_bf16_integer_exact(orc, seed=22):
    """bfloat16 holds the integers in [-256, 256] exactly; with integer inputs
    every partial sum is an integer below 2**53, so the product is exact."""
    rng = np.random.default_rng(seed)
    A = rng.integers(-200, 201, size=(2, 13, 150))
    B = rng.integers(-4, 5, size=(2, 9, 150))
    ref, absdot = orc.gemm_nt(bf16_bits(A), bf16_bits(B), dtype="bf16")
    assert np.array_equal(ref, np.einsum("bik,bjk->bij", A, B).astype(np.float64)), "bf16 integer product"
    assert np.array_equal(absdot, np.einsum("bik,bjk->bij", np.abs(A), np.abs(B)).astype(np.float64))


def f8_bits(x, dtype):
    """float64 values that the 8-bit format holds exactly -> uint8 bit patterns
    (through torch's casts; asserts the values are exact)."""
    import torch
    tt = torch.float8_e4m3fn if dtype == "e4m3" else torch.float8_e5m2
    t = torch.from_numpy(np.asarray(x, dtype=np.float64))
    q = t.to(tt)
    assert torch.equal(q.to(torch.float64), t), "value is not an %s" % dtype
    return q.view(torch.uint8).numpy().copy()


def pin_f8_decoders_exhaustive(orc):
    """All 256 patterns of each 8-bit format: E5M2 against the binary16 it is
    the upper byte of (numpy), E4M3 against torch's float8_e4m3fn cast."""
    bits = np.arange(256, dtype=np.uint16).astype(np.uint8)
    got = orc.f8_to_double(bits, "e5m2")
    want = (bits.astype(np.uint16) << 8).view(np.float16).astype(np.float64)
    n = np.isnan(want)
    assert np.array_equal(np.isnan(got), n) and np.array_equal(got[~n], want[~n]), "e5m2 decoder mismatch"
    import torch
    got = orc.f8_to_double(bits, "e4m3")
    want = torch.from_numpy(bits.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    n = np.isnan(want)
    assert np.array_equal(np.isnan(got), n), "e4m3 NaN patterns"
    assert np.array_equal(got[~n], want[~n]), "e4m3 decoder mismatch"
    assert np.array_equal(np.signbit(got[~n]), np.signbit(want[~n]))


def pin_f8_exact_tiny(orc, seed=31):
    """8-bit products over random tiny shapes, with subnormals and the formats'
    extremes, against exact rational sums; sampled = full."""
    rng = np.random.default_rng(seed)
    specials = {"e4m3": [0.0, -0.0, 2.0 ** -9, -(2.0 ** -6), 448.0, -448.0, 1.125, 3.5, 2.0 ** -7 * 5],
                "e5m2": [0.0, 2.0 ** -16, -(2.0 ** -14), 57344.0, -1.25, 0.75, 2.0 ** -15 * 3]}
    for dtype in ("e4m3", "e5m2"):
        vals = np.array(specials[dtype])
        for (batch, M, N, K) in ((1, 3, 4, 9), (2, 4, 3, 33)):
            a = rng.choice(vals, size=(batch, M, K))
            b = rng.choice(vals, size=(batch, N, K))
            A, B = f8_bits(a, dtype), f8_bits(b, dtype)
            ref, absdot = orc.gemm_nt(A, B, dtype=dtype)
            assert np.all(np.isfinite(ref)), "exact sums here are finite"
            g = gamma(max(K - 1, 0))
            for bi in range(batch):
                for i in range(M):
                    for j in range(N):
                        terms = [Fraction(float(a[bi, i, k])) * Fraction(float(b[bi, j, k])) for k in range(K)]
                        ex = sum(terms, Fraction(0))
                        exa = sum((abs(t) for t in terms), Fraction(0))
                        assert abs(Fraction(float(ref[bi, i, j])) - ex) <= Fraction(g) * exa * Fraction(1 + 2 * U) \
                            + Fraction(2 * U) * abs(ex) + Fraction(1, 2 ** 1074), "%s product" % dtype
                        assert abs(Fraction(float(absdot[bi, i, j])) - exa) <= Fraction(g + 2 * U) * exa \
                            + Fraction(1, 2 ** 1074), "%s absdot" % dtype
            bb = rng.integers(0, batch, size=12)
            ii = rng.integers(0, M, size=12)
            jj = rng.integers(0, N, size=12)
            sref, sabs = orc.gemm_nt_sampled(A, B, bb, ii, jj, dtype=dtype)
            assert np.array_equal(sref, ref[bb, ii, jj]) and np.array_equal(sabs, absdot[bb, ii, jj])


def pin_f8_integer_exact(orc, seed=32):
    """Integers in [-4, 4] are exact in both 8-bit formats; the products and
    sums are then exact integers."""
    rng = np.random.default_rng(seed)
    for dtype in ("e4m3", "e5m2"):
        A = rng.integers(-4, 5, size=(2, 11, 97))
        B = rng.integers(-4, 5, size=(2, 7, 97))
        ref, absdot = orc.gemm_nt(f8_bits(A, dtype), f8_bits(B, dtype), dtype=dtype)
        assert np.array_equal(ref, np.einsum("bik,bjk->bij", A, B).astype(np.float64)), "%s integers" % dtype
        assert np.array_equal(absdot, np.einsum("bik,bjk->bij", np.abs(A), np.abs(B)).astype(np.float64))


def pin_e8m0_decoder_exhaustive(orc):
    """All 256 E8M0 scale patterns: 2^(e-127) from math.ldexp, 255 is NaN."""
    import math
    bits = np.arange(256, dtype=np.uint16).astype(np.uint8)
    got = orc.e8m0_to_double(bits)
    want = np.array([math.ldexp(1.0, e - 127) for e in range(255)], dtype=np.float64)
    assert np.isnan(got[255]), "E8M0 255 is NaN"
    assert np.array_equal(got[:255], want), "E8M0 decoder mismatch"


def _mx_draw(rng, batch, rows, K, dtype, vals, lo=112, hi=142):
    x = rng.choice(vals, size=(batch, rows, K))
    s = rng.integers(lo, hi, size=(batch, rows, (K + 31) // 32)).astype(np.uint8)
    return x, f8_bits(x, dtype), s


def pin_mx_exact_tiny(orc, seed=41):
    """Block-scaled 8-bit products (K over several 32-element blocks and a
    partial one, random scales) against exact rational sums; sampled = full."""
    rng = np.random.default_rng(seed)
    specials = {"e4m3": [0.0, -0.0, 2.0 ** -9, -(2.0 ** -6), 448.0, -448.0, 1.125, 3.5, -0.75],
                "e5m2": [0.0, 2.0 ** -16, -(2.0 ** -14), 57344.0, -1.25, 0.75, 3.0]}
    for dtype in ("e4m3", "e5m2"):
        vals = np.array(specials[dtype])
        for (batch, M, N, K) in ((1, 3, 4, 40), (2, 2, 3, 97)):
            a, A, SA = _mx_draw(rng, batch, M, K, dtype, vals)
            b, B, SB = _mx_draw(rng, batch, N, K, dtype, vals)
            ref, absdot = orc.gemm_nt_mx(A, SA, B, SB, dtype=dtype)
            assert np.all(np.isfinite(ref)), "exact sums here are finite"
            g = gamma(max(K - 1, 0))
            for bi in range(batch):
                for i in range(M):
                    for j in range(N):
                        terms = [Fraction(float(a[bi, i, k])) * Fraction(2) ** (int(SA[bi, i, k // 32]) - 127)
                                 * Fraction(float(b[bi, j, k])) * Fraction(2) ** (int(SB[bi, j, k // 32]) - 127)
                                 for k in range(K)]
                        ex = sum(terms, Fraction(0))
                        exa = sum((abs(t) for t in terms), Fraction(0))
                        assert abs(Fraction(float(ref[bi, i, j])) - ex) <= Fraction(g) * exa * Fraction(1 + 2 * U) \
                            + Fraction(2 * U) * abs(ex) + Fraction(1, 2 ** 1074), "%s block-scaled product" % dtype
                        assert abs(Fraction(float(absdot[bi, i, j])) - exa) <= Fraction(g + 2 * U) * exa \
                            + Fraction(1, 2 ** 1074), "%s block-scaled absdot" % dtype
            bb = rng.integers(0, batch, size=12)
            ii = rng.integers(0, M, size=12)
            jj = rng.integers(0, N, size=12)
            sref, sabs = orc.gemm_nt_sampled_mx(A, SA, B, SB, bb, ii, jj, dtype=dtype)
            assert np.array_equal(sref, ref[bb, ii, jj]) and np.array_equal(sabs, absdot[bb, ii, jj])


def pin_mx_integer_exact(orc, seed=42):
    """Integers in [-4, 4] with scales 2^-3..2^3: every product and partial
    sum is exact, so the result equals numpy's einsum over the operands with
    each scale repeated over its 32 K elements, bit for bit."""
    rng = np.random.default_rng(seed)
    for dtype in ("e4m3", "e5m2"):
        batch, M, N, K = 2, 9, 7, 150
        A = rng.integers(-4, 5, size=(batch, M, K))
        B = rng.integers(-4, 5, size=(batch, N, K))
        SA = rng.integers(124, 131, size=(batch, M, (K + 31) // 32)).astype(np.uint8)
        SB = rng.integers(124, 131, size=(batch, N, (K + 31) // 32)).astype(np.uint8)
        ea = np.exp2(np.repeat(SA.astype(np.float64) - 127, 32, axis=2)[:, :, :K])
        eb = np.exp2(np.repeat(SB.astype(np.float64) - 127, 32, axis=2)[:, :, :K])
        want = np.einsum("bik,bjk->bij", A * ea, B * eb)
        ref, absdot = orc.gemm_nt_mx(f8_bits(A, dtype), SA, f8_bits(B, dtype), SB, dtype=dtype)
        assert np.array_equal(ref, want), "%s block-scaled integers" % dtype
        assert np.array_equal(absdot, np.einsum("bik,bjk->bij", np.abs(A) * ea, np.abs(B) * eb))


def pin_mx_unit_scales(orc, seed=43):
    """Scales of 127 (2^0) reduce the block-scaled product to the unscaled
    8-bit one, bit for bit; a scale of 128 on one whole row of A doubles that
    row of the result exactly."""
    rng = np.random.default_rng(seed)
    for dtype in ("e4m3", "e5m2"):
        x = rng.normal(0, 1, size=(3, 5, 70))
        A = f8_bits(torch_cast(x, dtype), dtype)
        B = f8_bits(torch_cast(rng.normal(0, 1, size=(3, 6, 70)), dtype), dtype)
        SA = np.full((3, 5, 3), 127, dtype=np.uint8)
        SB = np.full((3, 6, 3), 127, dtype=np.uint8)
        r1, a1 = orc.gemm_nt_mx(A, SA, B, SB, dtype=dtype)
        r0, a0 = orc.gemm_nt(A, B, dtype=dtype)
        assert np.array_equal(r1, r0) and np.array_equal(a1, a0), "%s unit scales" % dtype
        SA[1, 2, :] = 128
        r2, _ = orc.gemm_nt_mx(A, SA, B, SB, dtype=dtype)
        want = r0.copy()
        want[1, 2, :] *= 2
        assert np.array_equal(r2, want), "%s doubled row" % dtype


# 6- and 4-bit floats: (exponent bits, fraction bits, bias, total bits)
MINIFLOATS = {"e2m3": (2, 3, 1, 6), "e3m2": (3, 2, 3, 6), "e2m1": (2, 1, 1, 4)}


def minifloat_code(x, dtype):
    """Code of the value x in a 6- or 4-bit format, built from the format's
    field widths (exponent 0: subnormal fraction * 2^(1-bias-m)); x must be
    exactly representable."""
    e, m, b, n = MINIFLOATS[dtype]
    x = Fraction(x)
    sign = 1 if x < 0 else 0
    x = abs(x)
    for expo in range(2 ** e):
        for frac in range(2 ** m):
            v = (Fraction(frac, 2 ** m) * Fraction(2) ** (1 - b) if expo == 0
                 else (1 + Fraction(frac, 2 ** m)) * Fraction(2) ** (expo - b))
            if v == x:
                return (sign << (n - 1)) | (expo << m) | frac
    raise ValueError("%s is not an %s value" % (x, dtype))


def pin_f6f4_decoders(orc):
    """E2M3, E3M2 and E2M1, one per byte in its low bits: normal codes equal
    the binary16 of the same sign, fraction and unbiased exponent (numpy);
    the exponent-0 codes are equally spaced by 2^(1-bias-m) from 0; values
    increase with the code; the sign bit negates; the bits above the format
    are ignored; every value is an E4M3 value (torch's cast)."""
    import torch
    for dtype, (e, m, b, n) in MINIFLOATS.items():
        codes = np.arange(2 ** (n - 1), dtype=np.uint16).astype(np.uint8)
        v = orc.f8_to_double(codes, dtype)
        expo, frac = codes.astype(np.uint16) >> m, codes.astype(np.uint16) & (2 ** m - 1)
        normal = expo > 0
        h = (((expo.astype(np.int64) - b + 15) << 10) | (frac.astype(np.int64) << (10 - m))).astype(np.uint16)
        assert np.array_equal(v[normal], h[normal].view(np.float16).astype(np.float64)), "%s normal codes" % dtype
        sub = v[~normal]
        assert np.array_equal(sub, np.arange(2 ** m) * 2.0 ** (1 - b - m)), "%s subnormal codes" % dtype
        assert np.all(np.diff(v) > 0), "%s monotonic" % dtype
        neg = orc.f8_to_double(codes | np.uint8(1 << (n - 1)), dtype)
        assert np.array_equal(neg, -v) and np.all(np.signbit(neg)), "%s sign bit" % dtype
        hi = orc.f8_to_double(codes | np.uint8((0xff << n) & 0xff), dtype)
        assert np.array_equal(hi, v), "%s bits above the format" % dtype
        t = torch.from_numpy(v)
        assert torch.equal(t.to(torch.float8_e4m3fn).to(torch.float64), t), "%s values are E4M3 values" % dtype


def pin_f6f4_exact_tiny(orc, seed=51):
    """Products of random 6- and 4-bit codes (high bits set at random too)
    against exact rational sums of the decoded values, plain and
    block-scaled; sampled = full."""
    rng = np.random.default_rng(seed)
    for dtype in MINIFLOATS:
        for (batch, M, N, K) in ((1, 3, 4, 9), (2, 4, 3, 70)):
            A = rng.integers(0, 256, size=(batch, M, K)).astype(np.uint8)
            B = rng.integers(0, 256, size=(batch, N, K)).astype(np.uint8)
            a, b = orc.f8_to_double(A, dtype), orc.f8_to_double(B, dtype)
            SA = rng.integers(120, 135, size=(batch, M, (K + 31) // 32)).astype(np.uint8)
            SB = rng.integers(120, 135, size=(batch, N, (K + 31) // 32)).astype(np.uint8)
            for scaled in (False, True):
                ref, absdot = (orc.gemm_nt_mx(A, SA, B, SB, dtype=dtype) if scaled else orc.gemm_nt(A, B, dtype=dtype))
                g = gamma(max(K - 1, 0))
                for bi in range(batch):
                    for i in range(M):
                        for j in range(N):
                            terms = []
                            for k in range(K):
                                t = Fraction(float(a[bi, i, k])) * Fraction(float(b[bi, j, k]))
                                if scaled:
                                    t *= Fraction(2) ** (int(SA[bi, i, k // 32]) + int(SB[bi, j, k // 32]) - 254)
                                terms.append(t)
                            ex = sum(terms, Fraction(0))
                            exa = sum((abs(t) for t in terms), Fraction(0))
                            assert abs(Fraction(float(ref[bi, i, j])) - ex) <= Fraction(g) * exa * Fraction(1 + 2 * U) \
                                + Fraction(2 * U) * abs(ex) + Fraction(1, 2 ** 1074), "%s product" % dtype
                            assert abs(Fraction(float(absdot[bi, i, j])) - exa) <= Fraction(g + 2 * U) * exa \
                                + Fraction(1, 2 ** 1074), "%s absdot" % dtype
            bb = rng.integers(0, batch, size=12)
            ii = rng.integers(0, M, size=12)
            jj = rng.integers(0, N, size=12)
            sref, sabs = orc.gemm_nt_sampled(A, B, bb, ii, jj, dtype=dtype)
            ref, absdot = orc.gemm_nt(A, B, dtype=dtype)
            assert np.array_equal(sref, ref[bb, ii, jj]) and np.array_equal(sabs, absdot[bb, ii, jj])


def pin_f6f4_integer_exact(orc, seed=52):
    """Integers in [-4, 4], encoded from the field widths, give numpy's
    einsum exactly."""
    rng = np.random.default_rng(seed)
    for dtype in MINIFLOATS:
        A = rng.integers(-4, 5, size=(2, 7, 75))
        B = rng.integers(-4, 5, size=(2, 5, 75))
        enc = np.vectorize(lambda x: minifloat_code(int(x), dtype))
        ref, absdot = orc.gemm_nt(enc(A).astype(np.uint8), enc(B).astype(np.uint8), dtype=dtype)
        assert np.array_equal(ref, np.einsum("bik,bjk->bij", A, B).astype(np.float64)), "%s integers" % dtype
        assert np.array_equal(absdot, np.einsum("bik,bjk->bij", np.abs(A), np.abs(B)).astype(np.float64))


def torch_cast(x, dtype):
    """float64 values rounded to the nearest value of the 8-bit format."""
    import torch
    tt = torch.float8_e4m3fn if dtype == "e4m3" else torch.float8_e5m2
    return torch.from_numpy(np.asarray(x, dtype=np.float64)).to(tt).to(torch.float64).numpy()


ALL_PINS = [pin_decoder_exhaustive, pin_bruteforce_tiny, pin_k1_exact, pin_worked_examples,
            pin_closed_forms, pin_integer_exact, pin_numpy_crosscheck, pin_batched_and_sampled,
            pin_bf16_decoder_exhaustive, pin_bf16_exact_tiny, pin_bf16_integer_exact,
            pin_f8_decoders_exhaustive, pin_f8_exact_tiny, pin_f8_integer_exact,
            pin_e8m0_decoder_exhaustive, pin_mx_exact_tiny, pin_mx_integer_exact, pin_mx_unit_scales,
            pin_f6f4_decoders, pin_f6f4_exact_tiny, pin_f6f4_integer_exact]
