"""Python binding of libgemm_nt: Out = A @ B.T, fp16 inputs, fp32 accumulate/output.

The functions named like the C ABI (include/gemm_nt.h) take raw device
pointers and sizes and only marshal arguments; ``gemm_nt`` and
``gemm_nt_batched`` do the same for torch CUDA tensors (pointers, strides and
the current stream).  Every step of the product runs in the library's CUDA
kernels.  There is no fallback: if libgemm_nt.so has not been built, or a call
fails, an exception is raised.
"""
import ctypes
import enum
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libgemm_nt.so")


class Status(enum.IntEnum):
    OK = 0
    INVALID_VALUE = 1
    MISALIGNED = 2          # reserved: never returned
    OVERLAP = 3
    LAUNCH = 4
    DEVICE_TIMEOUT = 5
    UNSUPPORTED_DEVICE = 6
    NOT_SUPPORTED = 7
    SCRATCH_TOO_SMALL = 8


class DType(enum.IntEnum):
    F16 = 0
    BF16 = 1
    F32 = 2
    E4M3 = 3  # 8-bit floats (A and B only)
    E5M2 = 4
    E2M3 = 5  # 6- and 4-bit floats, packed along K, little-endian bits (A and B only)
    E3M2 = 6
    E2M1 = 7


class Major(enum.IntEnum):
    K = 0   # operand (rows, K) stored row-major
    MN = 1  # operand stored as its transpose, (K, rows) row-major


class Path(enum.IntEnum):
    AUTO = 0
    TC05 = 1
    SKINNY = 2
    MMASYNC = 3
    TC05_PAIR = 4
    TC05_M64 = 5   # 64-row tiles, plain M = 64 MMA
    TC05_WS = 6    # 32- or 64-row tiles, weight-stationary MMA


class GemmError(RuntimeError):
    def __init__(self, status):
        self.status = Status(status)
        super().__init__("libgemm_nt: %s (%s)" % (error_string(status), self.status.name))


# name -> (restype, argtypes); mirrors include/gemm_nt.h
_i64, _vp, _u64 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_uint64
_SIGNATURES = {
    "gemm_nt_f16_f32": (ctypes.c_int, [_vp, _vp, _vp] + [_i64] * 6 + [_vp]),
    "gemm_nt_f16_f32_batched": (ctypes.c_int, [_vp, _vp, _vp] + [_i64] * 10 + [_vp]),
    "gemm_nt_f16_f32_batched_path": (ctypes.c_int, [_vp, _vp, _vp] + [_i64] * 10 + [ctypes.c_int, _vp]),
    "gemm_nt_f16_f32_from_host": (ctypes.c_int, [_vp] * 6 + [_i64] * 4 + [_vp]),
    "gemm_nt_f16_f32_batched_no_alloc": (ctypes.c_int, [_vp, _vp, _vp] + [_i64] * 10 + [_vp]),
    "gemm_nt_batched_ex": (ctypes.c_int, [_vp, _vp, _vp, ctypes.c_int, ctypes.c_int] + [_i64] * 10
                           + [ctypes.c_int, _vp]),
    "gemm_nt_batched_major": (ctypes.c_int, [_vp, ctypes.c_int, _vp, ctypes.c_int, _vp, ctypes.c_int, ctypes.c_int]
                              + [_i64] * 10 + [ctypes.c_int, _vp]),
    "gemm_nt_mx": (ctypes.c_int, [_vp] * 5 + [ctypes.c_int, ctypes.c_int] + [_i64] * 10 + [ctypes.c_int, _vp]),
    "gemm_nt_mx_scale_bytes": (_i64, [_i64, _i64]),
    "gemm_nt_mx_pack_scales": (ctypes.c_int, [_vp, _i64, _i64, _vp, _i64, _i64, _i64, _vp]),
    "gemm_nt_select_path": (ctypes.c_int, [_vp, _vp, _vp] + [_i64] * 10),
    "gemm_nt_check": (ctypes.c_int, [_vp]),
    "gemm_nt_error_string": (ctypes.c_char_p, [ctypes.c_int]),
    "gemm_nt_probe_m16n8k16": (ctypes.c_int, [_vp] * 6),
    "gemm_nt_debug_set_wait_limit": (None, [_u64]),
    "gemm_nt_debug_set_fault": (None, [ctypes.c_int]),
}

_lib = None


def load(path=LIB_PATH):
    """Load libgemm_nt.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(
                "libgemm_nt.so is not built (%s); run `python -m dense_fp16_tensor_gemm_gb300._build`"
                % path)
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(status):
    if status != 0:
        raise GemmError(status)


def error_string(status):
    return load().gemm_nt_error_string(int(status)).decode()


# ---------------------------------------------------------------- C-ABI mirror
def gemm_nt_f16_f32(A, B, Out, M, N, K, lda, ldb, ldo, stream=0):
    _check(load().gemm_nt_f16_f32(A, B, Out, M, N, K, lda, ldb, ldo, stream))


def gemm_nt_f16_f32_batched(A, B, Out, M, N, K, lda, ldb, ldo, strideA, strideB, strideO, batch,
                            stream=0):
    _check(load().gemm_nt_f16_f32_batched(A, B, Out, M, N, K, lda, ldb, ldo, strideA, strideB,
                                          strideO, batch, stream))


def gemm_nt_f16_f32_batched_path(A, B, Out, M, N, K, lda, ldb, ldo, strideA, strideB, strideO,
                                 batch, path, stream=0):
    _check(load().gemm_nt_f16_f32_batched_path(A, B, Out, M, N, K, lda, ldb, ldo, strideA, strideB,
                                               strideO, batch, int(path), stream))


def gemm_nt_batched_ex(A, B, Out, ab_type, out_type, M, N, K, lda, ldb, ldo, strideA, strideB, strideO,
                       batch, path=0, stream=0):
    _check(load().gemm_nt_batched_ex(A, B, Out, int(ab_type), int(out_type), M, N, K, lda, ldb, ldo,
                                     strideA, strideB, strideO, batch, int(path), stream))


def gemm_nt_batched_major(A, a_major, B, b_major, Out, ab_type, out_type, M, N, K, lda, ldb, ldo, strideA,
                          strideB, strideO, batch, path=0, stream=0):
    _check(load().gemm_nt_batched_major(A, int(a_major), B, int(b_major), Out, int(ab_type), int(out_type), M, N,
                                        K, lda, ldb, ldo, strideA, strideB, strideO, batch, int(path), stream))


def gemm_nt_mx(A, SA, B, SB, Out, ab_type, out_type, M, N, K, lda, ldb, ldo, strideA, strideB, strideO, batch,
               path=0, stream=0):
    """Block-scaled 8-bit product; SA / SB in the packed atom layout (see
    include/gemm_nt.h)."""
    _check(load().gemm_nt_mx(A, SA, B, SB, Out, int(ab_type), int(out_type), M, N, K, lda, ldb, ldo, strideA,
                             strideB, strideO, batch, int(path), stream))


def gemm_nt_mx_scale_bytes(rows, K):
    return int(load().gemm_nt_mx_scale_bytes(rows, K))


def gemm_nt_mx_pack_scales(plain, ld, stride, packed, rows, K, batch=1, stream=0):
    _check(load().gemm_nt_mx_pack_scales(plain, ld, stride, packed, rows, K, batch, stream))


def gemm_nt_f16_f32_batched_no_alloc(A, B, Out, M, N, K, lda, ldb, ldo, strideA, strideB, strideO,
                                     batch, stream=0):
    """The batched product without any device allocation (fixed scratch array
    inside the library; see include/gemm_nt.h)."""
    _check(load().gemm_nt_f16_f32_batched_no_alloc(A, B, Out, M, N, K, lda, ldb, ldo, strideA, strideB,
                                                   strideO, batch, stream))


def gemm_nt_f16_f32_from_host(A_host, B_host, Out_host, dA, dB, dOut, M, N, K, batch, stream=0):
    _check(load().gemm_nt_f16_f32_from_host(A_host, B_host, Out_host, dA, dB, dOut, M, N, K, batch,
                                            stream))


def gemm_nt_select_path(A, B, Out, M, N, K, lda, ldb, ldo, strideA=0, strideB=0, strideO=0, batch=1):
    return Path(load().gemm_nt_select_path(A, B, Out, M, N, K, lda, ldb, ldo, strideA, strideB,
                                           strideO, batch))


def gemm_nt_check(stream=0):
    _check(load().gemm_nt_check(stream))


def gemm_nt_probe_m16n8k16(A, B, ar, br, dr, stream=0):
    _check(load().gemm_nt_probe_m16n8k16(A, B, ar, br, dr, stream))


def gemm_nt_debug_set_wait_limit(cycles):
    load().gemm_nt_debug_set_wait_limit(int(cycles))


def gemm_nt_debug_set_fault(fault):
    load().gemm_nt_debug_set_fault(int(fault))


# ---------------------------------------------------------------- torch tensors
def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _matrix_ld(t, name):
    if t.stride(-1) != 1:
        raise ValueError("%s must have unit stride along its last dimension" % name)
    return t.stride(-2) if t.shape[-2] > 1 else max(t.shape[-1], 1)


def _dtypes(A, B, out, out_dtype):
    import torch
    codes = {torch.float16: DType.F16, torch.bfloat16: DType.BF16, torch.float32: DType.F32,
             torch.float8_e4m3fn: DType.E4M3, torch.float8_e5m2: DType.E5M2}
    if A.dtype != B.dtype or A.dtype not in (torch.float16, torch.bfloat16, torch.float8_e4m3fn,
                                             torch.float8_e5m2):
        raise TypeError("A and B must have the same type: float16, bfloat16, float8_e4m3fn or float8_e5m2")
    dt = out.dtype if out is not None else (out_dtype or torch.float32)
    if dt not in (torch.float32, torch.float16, torch.bfloat16):
        raise TypeError("out must be float32, float16 or bfloat16")
    return codes[A.dtype], codes[dt], dt


def gemm_nt(A, B, out=None, path=Path.AUTO, stream=None, out_dtype=None):
    """Out = A @ B.T for torch CUDA tensors A (M,K), B (N,K), both fp16 or both
    bf16, accumulated in fp32.

    Row strides may exceed the row length; the last dimension must be
    contiguous.  ``out`` (M,N) is allocated if not given, as ``out_dtype``
    (default float32; float16 or bfloat16 round to nearest even).  Runs on
    ``stream`` (default: torch's current stream).
    """
    import torch
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[1]:
        raise ValueError("shapes: A (M,K), B (N,K)")
    ab, ot, dt = _dtypes(A, B, out, out_dtype)
    M, K = A.shape
    N = B.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=dt, device=A.device)
    if tuple(out.shape) != (M, N):
        raise ValueError("out must have shape (M,N)")
    gemm_nt_batched_ex(A.data_ptr(), B.data_ptr(), out.data_ptr(), ab, ot, M, N, K,
                       _matrix_ld(A, "A"), _matrix_ld(B, "B"), _matrix_ld(out, "out"),
                       0, 0, 0, 1, path, _stream_handle(stream))
    return out


def pack_mx_scales(S, K, stream=None):
    """Plain block scales -> the packed atom layout, on the device: S a uint8
    CUDA tensor (rows, ceil(K/32)) or (batch, rows, ceil(K/32)) of E8M0
    bytes, last dimension contiguous.  Returns a new uint8 tensor."""
    import torch
    if S.dtype != torch.uint8 or S.dim() not in (2, 3) or S.stride(-1) != 1:
        raise ValueError("S: uint8 (rows, ceil(K/32)) or (batch, rows, ceil(K/32)), last dimension contiguous")
    S3 = S if S.dim() == 3 else S[None]
    batch, rows, kb = S3.shape
    if kb != (K + 31) // 32:
        raise ValueError("S has %d scale columns, K=%d needs %d" % (kb, K, (K + 31) // 32))
    packed = torch.empty(batch * gemm_nt_mx_scale_bytes(rows, K), dtype=torch.uint8, device=S.device)
    gemm_nt_mx_pack_scales(S3.data_ptr(), S3.stride(1), S3.stride(0), packed.data_ptr(), rows, K, batch,
                           _stream_handle(stream))
    return packed


def gemm_nt_mx_tensors(A, SA, B, SB, out=None, path=Path.AUTO, stream=None, out_dtype=None):
    """Block-scaled Out = (A * sa) @ (B * sb).T for torch CUDA tensors: A (M,K)
    and B (N,K) both float8_e4m3fn or both float8_e5m2; SA (M, ceil(K/32))
    and SB (N, ceil(K/32)) uint8 E8M0 scales (2^(e-127)), one per 32
    consecutive K elements of a row, in the plain layout (packed here).
    ``out``/``out_dtype`` as in :func:`gemm_nt`."""
    import torch
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[1]:
        raise ValueError("shapes: A (M,K), B (N,K)")
    ab, ot, dt = _dtypes(A, B, out, out_dtype)
    if ab not in (DType.E4M3, DType.E5M2):
        raise TypeError("block-scaled inputs are float8_e4m3fn or float8_e5m2")
    M, K = A.shape
    N = B.shape[0]
    pa, pb = pack_mx_scales(SA, K, stream), pack_mx_scales(SB, K, stream)
    if out is None:
        out = torch.empty((M, N), dtype=dt, device=A.device)
    if tuple(out.shape) != (M, N):
        raise ValueError("out must have shape (M,N)")
    gemm_nt_mx(A.data_ptr(), pa.data_ptr(), B.data_ptr(), pb.data_ptr(), out.data_ptr(), ab, ot, M, N, K,
               _matrix_ld(A, "A"), _matrix_ld(B, "B"), _matrix_ld(out, "out"), 0, 0, 0, 1, path,
               _stream_handle(stream))
    return out


PACKED_BITS = {DType.E2M3: 6, DType.E3M2: 6, DType.E2M1: 4}


def gemm_nt_packed(A, B, K, ab_dtype, SA=None, SB=None, out=None, path=Path.AUTO, stream=None, out_dtype=None):
    """Out = A @ B.T for 6- or 4-bit float inputs stored packed: A (M, K*w/8)
    and B (N, K*w/8) uint8 CUDA tensors (w = 6 for E2M3 / E3M2, 4 for E2M1),
    element k of a row at bits [w*k, w*k+w) of the row, little-endian.  K is a
    multiple of 128, rows start on 32-byte boundaries.  With SA (M, K/32) and
    SB (N, K/32) uint8 E8M0 scales (plain layout) the product is block-scaled
    as in :func:`gemm_nt_mx_tensors`.  ``out``/``out_dtype`` as in :func:`gemm_nt`."""
    import torch
    ab = DType(ab_dtype)
    if ab not in PACKED_BITS:
        raise TypeError("ab_dtype must be E2M3, E3M2 or E2M1")
    bits = PACKED_BITS[ab]
    if A.dim() != 2 or B.dim() != 2 or A.dtype != torch.uint8 or B.dtype != torch.uint8:
        raise TypeError("A and B are 2-D uint8 tensors of packed elements")
    if K * bits % 8 or A.shape[1] != K * bits // 8 or B.shape[1] != K * bits // 8:
        raise ValueError("A and B must hold K packed elements per row")
    if (SA is None) != (SB is None):
        raise ValueError("give both SA and SB, or neither")
    dt = out.dtype if out is not None else (out_dtype or torch.float32)
    ocodes = {torch.float32: DType.F32, torch.float16: DType.F16, torch.bfloat16: DType.BF16}
    if dt not in ocodes:
        raise TypeError("out must be float32, float16 or bfloat16")
    M, N = A.shape[0], B.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=dt, device=A.device)
    if tuple(out.shape) != (M, N):
        raise ValueError("out must have shape (M,N)")
    # pitches in elements: the byte pitch of a row times 8 / w
    pa_bytes, pb_bytes = _matrix_ld(A, "A"), _matrix_ld(B, "B")
    if pa_bytes * 8 % bits or pb_bytes * 8 % bits:
        raise ValueError("row pitches must hold whole packing groups")
    lda, ldb = pa_bytes * 8 // bits, pb_bytes * 8 // bits
    if SA is None:
        gemm_nt_batched_ex(A.data_ptr(), B.data_ptr(), out.data_ptr(), ab, ocodes[dt], M, N, K, lda, ldb,
                           _matrix_ld(out, "out"), 0, 0, 0, 1, path, _stream_handle(stream))
    else:
        pa, pb = pack_mx_scales(SA, K, stream), pack_mx_scales(SB, K, stream)
        gemm_nt_mx(A.data_ptr(), pa.data_ptr(), B.data_ptr(), pb.data_ptr(), out.data_ptr(), ab, ocodes[dt], M, N,
                   K, lda, ldb, _matrix_ld(out, "out"), 0, 0, 0, 1, path, _stream_handle(stream))
    return out


def gemm_nt_batched(A, B, out=None, path=Path.AUTO, stream=None, out_dtype=None):
    """Out[b] = A[b] @ B[b].T for torch CUDA tensors A (batch,M,K), B (batch,N,K),
    both fp16 or both bf16 (a batch stride of 0, e.g. from ``expand``, shares
    the operand); ``out``/``out_dtype`` as in :func:`gemm_nt`."""
    import torch
    if A.dim() != 3 or B.dim() != 3 or A.shape[0] != B.shape[0] or A.shape[2] != B.shape[2]:
        raise ValueError("shapes: A (batch,M,K), B (batch,N,K)")
    ab, ot, dt = _dtypes(A, B, out, out_dtype)
    batch, M, K = A.shape
    N = B.shape[1]
    if out is None:
        out = torch.empty((batch, M, N), dtype=dt, device=A.device)
    if tuple(out.shape) != (batch, M, N):
        raise ValueError("out must have shape (batch,M,N)")
    gemm_nt_batched_ex(A.data_ptr(), B.data_ptr(), out.data_ptr(), ab, ot, M, N, K,
                       _matrix_ld(A, "A"), _matrix_ld(B, "B"), _matrix_ld(out, "out"),
                       A.stride(0), B.stride(0), out.stride(0), batch, path, _stream_handle(stream))
    return out
