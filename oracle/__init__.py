"""CPU oracle for Out = A @ B.T (fp16 inputs), accumulated in double.

TEST INFRASTRUCTURE ONLY: imported by tests/, by the package smoke check and
by the benchmark's CPU-baseline leg.  The CUDA library never imports, links or
executes anything here, and nothing here imports the CUDA library.

The arithmetic lives in ``gemm_oracle.c`` (plain C, IEEE double, sequential k):
    ref[b,i,j]    = sum_k dbl(A[b,i,k]) * dbl(B[b,j,k])
    absdot[b,i,j] = sum_k |dbl(A[b,i,k]) * dbl(B[b,j,k])|
following "Warp Matrix Instructions" (opening paragraph: Out = A @ B.T, float16
inputs, float32 accumulation) and "Blackwell Tensor Cores", section "The
Accumulator's Lifetime" (the same product with a TMEM float32 accumulator);
double replaces float32 as the accumulator so the oracle is at least as
accurate as any fp32 implementation.

The same product for bfloat16 inputs ("Warp Matrix Instructions", "Other
Fragment Shapes and Transfers") is ``gemm_nt(..., dtype="bf16")``, with inputs
given as uint16 bit patterns; for the 8-bit floats E4M3 and E5M2 it is
``dtype="e4m3"`` / ``"e5m2"`` with uint8 bit patterns, and for the 6- and
4-bit floats E2M3, E3M2 and E2M1 (one per byte, in its low bits)
``dtype="e2m3"`` / ``"e3m2"`` / ``"e2m1"``.  The block-scaled form
(one E8M0 power-of-two scale per 32 consecutive K elements of every row of A
and of B; "Blackwell Tensor Cores" names block scaling and its tcgen05.cp
scale operands without a formula, and the plain microscaling reading is taken)
is ``gemm_nt_mx``.

Parity rule used by the tests (stated once here so every test uses the same):
    |Out - ref| <= 1e-3 * absdot + 1e-6    elementwise, and
    Out == ref exactly when every partial sum is an integer below 2**24.
A 16-bit Out adds the rounding of ref into its format (half a unit in the
last place: 2**-11 relative for float16, 2**-8 for bfloat16), and in the exact
case Out == round_output(ref) exactly.
"""
import ctypes

import numpy as np

from . import build as _build


def _u16(x):
    x = np.asarray(x)
    if x.dtype == np.float16:
        x = x.view(np.uint16)
    if x.dtype != np.uint16:
        raise TypeError("oracle inputs must be float16 (or their uint16 bit patterns)")
    return np.ascontiguousarray(x)


F8_TYPES = ("e4m3", "e5m2", "e2m3", "e3m2", "e2m1")
# 8-bit container formats: codes of the oracle's dec8 (those of the MMA's
# instruction descriptor); E2M3 / E3M2 sit in the low 6 bits of a byte, E2M1 in
# the low 4
FMT8 = {"e4m3": 0, "e5m2": 1, "e2m3": 3, "e3m2": 4, "e2m1": 5}


def _u8(x):
    x = np.asarray(x)
    if x.dtype != np.uint8:
        raise TypeError("8-bit float inputs are given as uint8 bit patterns")
    return np.ascontiguousarray(x)


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


class Oracle:
    """ctypes view of one build of gemm_oracle.c (the default build, or a test's
    deliberately broken copy used to show that the pins catch mistakes)."""

    def __init__(self, path):
        lib = ctypes.CDLL(path)
        i64, u16p, f64p, i64p = (ctypes.c_int64, ctypes.POINTER(ctypes.c_uint16),
                                 ctypes.POINTER(ctypes.c_double),
                                 ctypes.POINTER(ctypes.c_int64))
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_half_to_double.restype = ctypes.c_double
        lib.oracle_half_to_double_array.argtypes = [u16p, f64p, i64]
        lib.oracle_half_to_double_array.restype = None
        lib.oracle_gemm_nt.argtypes = [u16p, u16p, f64p, f64p] + [i64] * 10 + [ctypes.c_int]
        lib.oracle_gemm_nt.restype = None
        lib.oracle_gemm_nt_sampled.argtypes = [u16p, u16p, i64p, i64p, i64p, i64, i64, i64, i64,
                                               i64, i64, f64p, f64p, ctypes.c_int]
        lib.oracle_gemm_nt_sampled.restype = None
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = ctypes.c_int
        self.has_bf16 = hasattr(lib, "oracle_gemm_nt_bf16")
        if self.has_bf16:
            lib.oracle_bf16_to_double_array.argtypes = [u16p, f64p, i64]
            lib.oracle_bf16_to_double_array.restype = None
            lib.oracle_gemm_nt_bf16.argtypes = lib.oracle_gemm_nt.argtypes
            lib.oracle_gemm_nt_bf16.restype = None
            lib.oracle_gemm_nt_sampled_bf16.argtypes = lib.oracle_gemm_nt_sampled.argtypes
            lib.oracle_gemm_nt_sampled_bf16.restype = None
        self.has_f8 = hasattr(lib, "oracle_gemm_nt_f8")
        if self.has_f8:
            u8p = ctypes.POINTER(ctypes.c_uint8)
            lib.oracle_f8_to_double_array.argtypes = [u8p, f64p, i64, ctypes.c_int]
            lib.oracle_f8_to_double_array.restype = None
            lib.oracle_gemm_nt_f8.argtypes = [u8p, u8p, f64p, f64p] + [i64] * 10 + [ctypes.c_int, ctypes.c_int]
            lib.oracle_gemm_nt_f8.restype = None
            lib.oracle_gemm_nt_sampled_f8.argtypes = [u8p, u8p, i64p, i64p, i64p, i64, i64, i64, i64, i64, i64,
                                                      f64p, f64p, ctypes.c_int, ctypes.c_int]
            lib.oracle_gemm_nt_sampled_f8.restype = None
        self.has_mx = hasattr(lib, "oracle_gemm_nt_mx")
        if self.has_mx:
            u8p = ctypes.POINTER(ctypes.c_uint8)
            lib.oracle_e8m0_to_double_array.argtypes = [u8p, f64p, i64]
            lib.oracle_e8m0_to_double_array.restype = None
            lib.oracle_gemm_nt_mx.argtypes = [u8p, u8p, u8p, u8p, f64p, f64p] + [i64] * 14 + [ctypes.c_int] * 2
            lib.oracle_gemm_nt_mx.restype = None
            lib.oracle_gemm_nt_sampled_mx.argtypes = ([u8p] * 4 + [i64p] * 3 + [i64] * 10 + [f64p, f64p]
                                                      + [ctypes.c_int] * 2)
            lib.oracle_gemm_nt_sampled_mx.restype = None
        self.lib = lib
        self.path = path

    def max_threads(self) -> int:
        """Threads the oracle's OpenMP loops use by default."""
        return int(self.lib.oracle_max_threads())

    def half_to_double(self, bits) -> np.ndarray:
        """Decode fp16 values (float16 array or uint16 bit patterns) to float64."""
        b = _u16(bits)
        out = np.empty(b.shape, dtype=np.float64)
        self.lib.oracle_half_to_double_array(_ptr(b, ctypes.c_uint16),
                                             _ptr(out, ctypes.c_double), b.size)
        return out

    def bf16_to_double(self, bits) -> np.ndarray:
        """Decode bfloat16 bit patterns (uint16) to float64."""
        b = np.ascontiguousarray(bits, dtype=np.uint16)
        out = np.empty(b.shape, dtype=np.float64)
        self.lib.oracle_bf16_to_double_array(_ptr(b, ctypes.c_uint16), _ptr(out, ctypes.c_double), b.size)
        return out

    def f8_to_double(self, bits, dtype: str) -> np.ndarray:
        """Decode 8-bit container patterns (uint8; dtype one of F8_TYPES) to float64."""
        b = np.ascontiguousarray(bits, dtype=np.uint8)
        out = np.empty(b.shape, dtype=np.float64)
        self.lib.oracle_f8_to_double_array(_ptr(b, ctypes.c_uint8), _ptr(out, ctypes.c_double), b.size,
                                           FMT8[dtype])
        return out

    def gemm_nt(self, A, B, nthreads: int = 0, dtype: str = "f16"):
        """Full product.  A: (M,K) or (batch,M,K); B: (N,K) or (batch,N,K);
        float16 arrays, or bit patterns: uint16 for fp16 (dtype "f16") and
        bfloat16 ("bf16"), uint8 for the 8-bit floats "e4m3" and "e5m2".

        Returns (ref, absdot), float64 arrays of shape (M,N) or (batch,M,N).
        """
        if dtype in F8_TYPES:
            return self._gemm_nt_f8(A, B, nthreads, dtype)
        fn = self._fn("oracle_gemm_nt", dtype)
        a, b = _u16(A), _u16(B)
        squeeze = a.ndim == 2
        if squeeze:
            a, b = a[None], b[None]
        if a.ndim != 3 or b.ndim != 3 or a.shape[0] != b.shape[0] or a.shape[2] != b.shape[2]:
            raise ValueError("shape mismatch: A %s, B %s" % (np.shape(A), np.shape(B)))
        batch, M, K = a.shape
        N = b.shape[1]
        ref = np.empty((batch, M, N), dtype=np.float64)
        absdot = np.empty((batch, M, N), dtype=np.float64)
        fn(_ptr(a, ctypes.c_uint16), _ptr(b, ctypes.c_uint16),
           _ptr(ref, ctypes.c_double), _ptr(absdot, ctypes.c_double),
           batch, M, N, K, K, K, N, M * K, N * K, M * N, int(nthreads))
        if squeeze:
            ref, absdot = ref[0], absdot[0]
        return ref, absdot

    def _gemm_nt_f8(self, A, B, nthreads, dtype):
        if not self.has_f8:
            raise ValueError("this oracle build has no 8-bit float product")
        a, b = _u8(A), _u8(B)
        squeeze = a.ndim == 2
        if squeeze:
            a, b = a[None], b[None]
        if a.ndim != 3 or b.ndim != 3 or a.shape[0] != b.shape[0] or a.shape[2] != b.shape[2]:
            raise ValueError("shape mismatch: A %s, B %s" % (np.shape(A), np.shape(B)))
        batch, M, K = a.shape
        N = b.shape[1]
        ref = np.empty((batch, M, N), dtype=np.float64)
        absdot = np.empty((batch, M, N), dtype=np.float64)
        self.lib.oracle_gemm_nt_f8(_ptr(a, ctypes.c_uint8), _ptr(b, ctypes.c_uint8), _ptr(ref, ctypes.c_double),
                                   _ptr(absdot, ctypes.c_double), batch, M, N, K, K, K, N, M * K, N * K, M * N,
                                   int(nthreads), FMT8[dtype])
        if squeeze:
            ref, absdot = ref[0], absdot[0]
        return ref, absdot

    def e8m0_to_double(self, bits) -> np.ndarray:
        """Decode E8M0 scales (uint8: 2^(e-127), 255 = NaN) to float64."""
        b = np.ascontiguousarray(bits, dtype=np.uint8)
        out = np.empty(b.shape, dtype=np.float64)
        self.lib.oracle_e8m0_to_double_array(_ptr(b, ctypes.c_uint8), _ptr(out, ctypes.c_double), b.size)
        return out

    def _mx_operands(self, A, SA, B, SB):
        if not self.has_mx:
            raise ValueError("this oracle build has no block-scaled product")
        a, b, sa, sb = _u8(A), _u8(B), _u8(SA), _u8(SB)
        if a.ndim == 2:
            a, b, sa, sb = a[None], b[None], sa[None], sb[None]
        batch, M, K = a.shape
        N = b.shape[1]
        kb = (K + 31) // 32
        if (b.shape != (batch, N, K) or sa.shape != (batch, M, kb) or sb.shape != (batch, N, kb)):
            raise ValueError("shape mismatch: A %s, SA %s, B %s, SB %s"
                             % (np.shape(A), np.shape(SA), np.shape(B), np.shape(SB)))
        return a, sa, b, sb

    def gemm_nt_mx(self, A, SA, B, SB, nthreads: int = 0, dtype: str = "e4m3"):
        """Block-scaled product.  A (M,K) or (batch,M,K) and B (N,K) or
        (batch,N,K): uint8 patterns of dtype "e4m3" or "e5m2"; SA (.., M,
        ceil(K/32)) and SB (.., N, ceil(K/32)): uint8 E8M0 scales, one per 32
        consecutive K elements of a row.  Returns (ref, absdot), float64."""
        squeeze = np.ndim(A) == 2
        a, sa, b, sb = self._mx_operands(A, SA, B, SB)
        batch, M, K = a.shape
        N, kb = b.shape[1], sa.shape[2]
        ref = np.empty((batch, M, N), dtype=np.float64)
        absdot = np.empty((batch, M, N), dtype=np.float64)
        self.lib.oracle_gemm_nt_mx(_ptr(a, ctypes.c_uint8), _ptr(sa, ctypes.c_uint8), _ptr(b, ctypes.c_uint8),
                                   _ptr(sb, ctypes.c_uint8), _ptr(ref, ctypes.c_double), _ptr(absdot, ctypes.c_double),
                                   batch, M, N, K, K, K, kb, kb, N, M * K, N * K, M * kb, N * kb, M * N,
                                   int(nthreads), FMT8[dtype])
        if squeeze:
            ref, absdot = ref[0], absdot[0]
        return ref, absdot

    def gemm_nt_sampled_mx(self, A, SA, B, SB, bidx, iidx, jidx, nthreads: int = 0, dtype: str = "e4m3"):
        """Selected elements of :meth:`gemm_nt_mx` (2-D inputs take bidx = 0)."""
        a, sa, b, sb = self._mx_operands(A, SA, B, SB)
        batch, M, K = a.shape
        N, kb = b.shape[1], sa.shape[2]
        ii = np.ascontiguousarray(iidx, dtype=np.int64)
        jj = np.ascontiguousarray(jidx, dtype=np.int64)
        bb = np.ascontiguousarray(np.broadcast_to(np.asarray(bidx, dtype=np.int64), ii.shape))
        if ii.shape != jj.shape:
            raise ValueError("index arrays differ in shape")
        if ii.size and (ii.min() < 0 or ii.max() >= M or jj.min() < 0 or jj.max() >= N
                        or bb.min() < 0 or bb.max() >= batch):
            raise IndexError("sample index out of range")
        ref = np.empty(ii.shape, dtype=np.float64)
        absdot = np.empty(ii.shape, dtype=np.float64)
        self.lib.oracle_gemm_nt_sampled_mx(
            _ptr(a, ctypes.c_uint8), _ptr(sa, ctypes.c_uint8), _ptr(b, ctypes.c_uint8), _ptr(sb, ctypes.c_uint8),
            _ptr(bb, ctypes.c_int64), _ptr(ii, ctypes.c_int64), _ptr(jj, ctypes.c_int64), ii.size, K, K, K, kb, kb,
            M * K, N * K, M * kb, N * kb, _ptr(ref, ctypes.c_double), _ptr(absdot, ctypes.c_double), int(nthreads),
            FMT8[dtype])
        return ref, absdot

    def _fn(self, name, dtype):
        if dtype == "f16":
            return getattr(self.lib, name)
        if dtype == "bf16" and self.has_bf16:
            return getattr(self.lib, name + "_bf16")
        raise ValueError("unknown input type %r" % dtype)

    def gemm_nt_sampled(self, A, B, bidx, iidx, jidx, nthreads: int = 0, dtype: str = "f16"):
        """Selected elements (bidx[s], iidx[s], jidx[s]) of the product.

        A, B as in :meth:`gemm_nt` (2-D inputs take bidx = 0).  Returns
        (ref, absdot), float64 arrays of length len(iidx).
        """
        f8 = dtype in F8_TYPES
        a, b = (_u8(A), _u8(B)) if f8 else (_u16(A), _u16(B))
        if a.ndim == 2:
            a, b = a[None], b[None]
        batch, M, K = a.shape
        N = b.shape[1]
        ii = np.ascontiguousarray(iidx, dtype=np.int64)
        jj = np.ascontiguousarray(jidx, dtype=np.int64)
        bb = np.ascontiguousarray(np.broadcast_to(np.asarray(bidx, dtype=np.int64), ii.shape))
        if ii.shape != jj.shape:
            raise ValueError("index arrays differ in shape")
        if ii.size and (ii.min() < 0 or ii.max() >= M or jj.min() < 0 or jj.max() >= N
                        or bb.min() < 0 or bb.max() >= batch):
            raise IndexError("sample index out of range")
        ref = np.empty(ii.shape, dtype=np.float64)
        absdot = np.empty(ii.shape, dtype=np.float64)
        if f8:
            self.lib.oracle_gemm_nt_sampled_f8(
                _ptr(a, ctypes.c_uint8), _ptr(b, ctypes.c_uint8), _ptr(bb, ctypes.c_int64),
                _ptr(ii, ctypes.c_int64), _ptr(jj, ctypes.c_int64), ii.size, K, K, K, M * K, N * K,
                _ptr(ref, ctypes.c_double), _ptr(absdot, ctypes.c_double), int(nthreads),
                FMT8[dtype])
            return ref, absdot
        self._fn("oracle_gemm_nt_sampled", dtype)(
            _ptr(a, ctypes.c_uint16), _ptr(b, ctypes.c_uint16), _ptr(bb, ctypes.c_int64),
            _ptr(ii, ctypes.c_int64), _ptr(jj, ctypes.c_int64), ii.size, K, K, K, M * K, N * K,
            _ptr(ref, ctypes.c_double), _ptr(absdot, ctypes.c_double), int(nthreads))
        return ref, absdot


_default = None


def default() -> Oracle:
    """The oracle built from oracle/gemm_oracle.c (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle(_build.build())
    return _default


def max_threads() -> int:
    return default().max_threads()


def half_to_double(bits):
    return default().half_to_double(bits)


def bf16_to_double(bits):
    return default().bf16_to_double(bits)


def f8_to_double(bits, dtype):
    return default().f8_to_double(bits, dtype)


def gemm_nt(A, B, nthreads: int = 0, dtype: str = "f16"):
    return default().gemm_nt(A, B, nthreads, dtype)


def e8m0_to_double(bits):
    return default().e8m0_to_double(bits)


def gemm_nt_mx(A, SA, B, SB, nthreads: int = 0, dtype: str = "e4m3"):
    return default().gemm_nt_mx(A, SA, B, SB, nthreads, dtype)


def gemm_nt_sampled_mx(A, SA, B, SB, bidx, iidx, jidx, nthreads: int = 0, dtype: str = "e4m3"):
    return default().gemm_nt_sampled_mx(A, SA, B, SB, bidx, iidx, jidx, nthreads, dtype)


def gemm_nt_sampled(A, B, bidx, iidx, jidx, nthreads: int = 0, dtype: str = "f16"):
    return default().gemm_nt_sampled(A, B, bidx, iidx, jidx, nthreads, dtype)


# Half the spacing of an output format relative to the value (the largest
# error of rounding to nearest), and half its smallest subnormal.
OUT_ROUNDING = {"f32": (2.0 ** -24, 2.0 ** -150), "f16": (2.0 ** -11, 2.0 ** -25),
                "bf16": (2.0 ** -8, 2.0 ** -134)}


def round_output(ref, out_dtype: str):
    """The value a ``out_dtype`` Out element holds when the fp32 accumulator
    equals ``ref`` exactly (integer inputs with partial sums below 2**24): ref
    rounded once to nearest, ties to even, in that format; float64 result.

    float16: numpy's float32 -> float16 cast.  bfloat16: written out on the
    binary32 bits -- add 0x7FFF plus the lowest kept bit, keep the upper 16."""
    r = np.asarray(ref, dtype=np.float64)
    f = r.astype(np.float32)
    if not np.array_equal(f.astype(np.float64), r, equal_nan=True):
        raise ValueError("round_output needs results that float32 holds exactly")
    if out_dtype == "f32":
        return f.astype(np.float64)
    if out_dtype == "f16":
        return f.astype(np.float16).astype(np.float64)
    if out_dtype == "bf16":
        u = np.ascontiguousarray(f).view(np.uint32).astype(np.uint64)
        kept = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
        return kept.astype(np.uint32).view(np.float32).astype(np.float64)
    raise ValueError("unknown output type %r" % out_dtype)


def within_tolerance(out, ref, absdot, out_dtype: str = "f32"):
    """Elementwise parity predicate |out-ref| <= 1e-3*absdot + 1e-6, widened
    for a 16-bit Out by the rounding of ref into that format."""
    out = np.asarray(out, dtype=np.float64)
    tol = 1e-3 * absdot + 1e-6
    if out_dtype != "f32":
        rel, tiny = OUT_ROUNDING[out_dtype]
        tol = tol + rel * np.abs(ref) + tiny
    return np.abs(out - ref) <= tol
