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

Parity rule used by the tests (stated once here so every test uses the same):
    |Out - ref| <= 1e-3 * absdot + 1e-6    elementwise, and
    Out == ref exactly when every partial sum is an integer below 2**24.
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

    def gemm_nt(self, A, B, nthreads: int = 0):
        """Full product.  A: (M,K) or (batch,M,K) fp16; B: (N,K) or (batch,N,K).

        Returns (ref, absdot), float64 arrays of shape (M,N) or (batch,M,N).
        """
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
        self.lib.oracle_gemm_nt(_ptr(a, ctypes.c_uint16), _ptr(b, ctypes.c_uint16),
                                _ptr(ref, ctypes.c_double), _ptr(absdot, ctypes.c_double),
                                batch, M, N, K, K, K, N, M * K, N * K, M * N, int(nthreads))
        if squeeze:
            ref, absdot = ref[0], absdot[0]
        return ref, absdot

    def gemm_nt_sampled(self, A, B, bidx, iidx, jidx, nthreads: int = 0):
        """Selected elements (bidx[s], iidx[s], jidx[s]) of the product.

        A, B as in :meth:`gemm_nt` (2-D inputs take bidx = 0).  Returns
        (ref, absdot), float64 arrays of length len(iidx).
        """
        a, b = _u16(A), _u16(B)
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
        self.lib.oracle_gemm_nt_sampled(_ptr(a, ctypes.c_uint16), _ptr(b, ctypes.c_uint16),
                                        _ptr(bb, ctypes.c_int64), _ptr(ii, ctypes.c_int64),
                                        _ptr(jj, ctypes.c_int64), ii.size, K, K, K, M * K, N * K,
                                        _ptr(ref, ctypes.c_double), _ptr(absdot, ctypes.c_double),
                                        int(nthreads))
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


def gemm_nt(A, B, nthreads: int = 0):
    return default().gemm_nt(A, B, nthreads)


def gemm_nt_sampled(A, B, bidx, iidx, jidx, nthreads: int = 0):
    return default().gemm_nt_sampled(A, B, bidx, iidx, jidx, nthreads)


def within_tolerance(out, ref, absdot):
    """Elementwise parity predicate |out-ref| <= 1e-3*absdot + 1e-6."""
    out = np.asarray(out, dtype=np.float64)
    return np.abs(out - ref) <= 1e-3 * absdot + 1e-6
