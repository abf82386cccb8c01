"""The C ABI without a GPU: the library builds and loads, exports every
function include/gemm_nt.h declares, and rejects bad arguments on the host
before any CUDA call."""
import ctypes
import os
import re

import pytest

import dense_fp16_tensor_gemm_gb300 as gnt
from dense_fp16_tensor_gemm_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm_nt.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return gnt.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("gemm_nt_f16_f32", "gemm_nt_f16_f32_batched", "gemm_nt_check",
              "gemm_nt_error_string", "gemm_nt_select_path"):
        assert n in names


def _declaration(name):
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    m = re.search(r"\b%s\s*\(([^)]*)\)" % name, text)
    assert m, name
    return [p.split()[-1].lstrip("*") for p in m.group(1).split(",")]


def test_boundary_signatures():
    """The plain and batched products take (A, B, Out), the sizes, the leading
    dimensions, then (batched) the three batch strides and the batch count,
    then the stream; every other batched entry point keeps that order."""
    assert _declaration("gemm_nt_f16_f32") == ["A", "B", "Out", "M", "N", "K", "lda", "ldb", "ldo", "stream"]
    assert _declaration("gemm_nt_f16_f32_batched") == [
        "A", "B", "Out", "M", "N", "K", "lda", "ldb", "ldo", "strideA", "strideB", "strideO", "batch", "stream"]
    assert _declaration("gemm_nt_check") == ["stream"]
    assert _declaration("gemm_nt_error_string") == ["status"]
    for name in ("gemm_nt_f16_f32_batched_path", "gemm_nt_batched_ex", "gemm_nt_batched_major", "gemm_nt_mx",
                 "gemm_nt_f16_f32_batched_no_alloc", "gemm_nt_select_path"):
        args = _declaration(name)
        i = args.index("ldo")
        assert args[i + 1:i + 5] == ["strideA", "strideB", "strideO", "batch"], name


def _header_enum(name):
    text = open(HEADER).read()
    body = re.search(r"typedef enum %s \{(.*?)\}" % name, text, flags=re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    return {k: int(v) for k, v in re.findall(r"([A-Z0-9_]+)\s*=\s*(-?\d+)", body)}


def test_status_codes():
    """Status values of the boundary, and the binding mirrors the header."""
    codes = _header_enum("gemm_status")
    assert {k: codes[k] for k in ("GEMM_OK", "GEMM_ERR_INVALID_VALUE", "GEMM_ERR_MISALIGNED", "GEMM_ERR_OVERLAP",
                                  "GEMM_ERR_LAUNCH", "GEMM_ERR_DEVICE_TIMEOUT",
                                  "GEMM_ERR_UNSUPPORTED_DEVICE")} == {
        "GEMM_OK": 0, "GEMM_ERR_INVALID_VALUE": 1, "GEMM_ERR_MISALIGNED": 2, "GEMM_ERR_OVERLAP": 3,
        "GEMM_ERR_LAUNCH": 4, "GEMM_ERR_DEVICE_TIMEOUT": 5, "GEMM_ERR_UNSUPPORTED_DEVICE": 6}
    mirrored = {("GEMM_OK" if s.name == "OK" else "GEMM_ERR_" + s.name): int(s) for s in gnt.Status}
    assert mirrored == codes
    for enum_name, py in (("gemm_dtype", gnt.DType), ("gemm_path", gnt.Path), ("gemm_major", gnt.Major)):
        prefix = {"gemm_dtype": "GEMM_DTYPE_", "gemm_path": "GEMM_PATH_", "gemm_major": "GEMM_MAJOR_"}[enum_name]
        assert {prefix + m.name: int(m) for m in py} == _header_enum(enum_name), enum_name


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) <= set(gnt._SIGNATURES)


def test_error_strings(lib):
    texts = [gnt.error_string(s) for s in gnt.Status]
    assert all(texts) and len(set(texts)) == len(texts)
    assert "unknown status" not in texts
    assert gnt.error_string(99) == "unknown status"
    assert gnt.error_string(-1) == "unknown status"


FAKE_A, FAKE_B, FAKE_O = 0x10000000, 0x20000000, 0x30000000


@pytest.mark.parametrize("args,status", [
    ((FAKE_A, FAKE_B, FAKE_O, -1, 8, 8, 8, 8, 8), gnt.Status.INVALID_VALUE),
    ((FAKE_A, FAKE_B, FAKE_O, 8, 8, 8, 7, 8, 8), gnt.Status.INVALID_VALUE),   # lda < K
    ((FAKE_A, FAKE_B, FAKE_O, 8, 8, 8, 8, 7, 8), gnt.Status.INVALID_VALUE),   # ldb < K
    ((FAKE_A, FAKE_B, FAKE_O, 8, 8, 8, 8, 8, 7), gnt.Status.INVALID_VALUE),   # ldo < N
    ((0, FAKE_B, FAKE_O, 8, 8, 8, 8, 8, 8), gnt.Status.INVALID_VALUE),        # null A
    ((FAKE_A, FAKE_B, 0, 8, 8, 8, 8, 8, 8), gnt.Status.INVALID_VALUE),        # null Out
    ((FAKE_A, FAKE_B, FAKE_O + 2, 8, 8, 8, 8, 8, 8), gnt.Status.INVALID_VALUE),  # Out not 4-aligned
    ((FAKE_A, FAKE_B, FAKE_A + 64, 8, 8, 8, 8, 8, 8), gnt.Status.OVERLAP),    # Out inside A
    ((FAKE_A, FAKE_B, FAKE_B - 16, 8, 8, 8, 8, 8, 8), gnt.Status.OVERLAP),    # Out runs into B
    ((FAKE_A, FAKE_B, FAKE_O, 2 ** 31, 8, 8, 8, 8, 8), gnt.Status.INVALID_VALUE),
])
def test_host_validation(lib, args, status):
    assert lib.gemm_nt_f16_f32(*args, None) == status


def test_empty_problems_launch_nothing(lib):
    # M, N or batch zero: success without touching the (absent) device
    assert lib.gemm_nt_f16_f32(FAKE_A, FAKE_B, FAKE_O, 0, 8, 8, 8, 8, 8, None) == 0
    assert lib.gemm_nt_f16_f32(0, 0, 0, 8, 0, 8, 8, 8, 8, None) == 0
    assert lib.gemm_nt_f16_f32_batched(FAKE_A, FAKE_B, FAKE_O, 8, 8, 8, 8, 8, 8, 64, 64, 64, 0,
                                       None) == 0


def test_batched_validation(lib):
    f = lib.gemm_nt_f16_f32_batched
    # batches of Out overlap (strideO too small)
    assert f(FAKE_A, FAKE_B, FAKE_O, 8, 8, 8, 8, 8, 8, 64, 64, 63, 2, None) == gnt.Status.OVERLAP
    # negative stride
    assert f(FAKE_A, FAKE_B, FAKE_O, 8, 8, 8, 8, 8, 8, -64, 64, 64, 2, None) == gnt.Status.INVALID_VALUE
    # bad explicit path
    for bad in (99, 7, -1):
        assert lib.gemm_nt_f16_f32_batched_path(FAKE_A, FAKE_B, FAKE_O, 8, 8, 8, 8, 8, 8, 0, 0, 0, 1, bad,
                                                None) == gnt.Status.INVALID_VALUE
    # the path numbers of the header
    assert [int(x) for x in gnt.Path] == list(range(7))


def test_from_host_validation(lib):
    f = lib.gemm_nt_f16_f32_from_host
    assert f(FAKE_A, FAKE_B, FAKE_O, FAKE_A, FAKE_B, 0, 8, 8, 8, 1, None) == gnt.Status.INVALID_VALUE
    assert f(0, 0, 0, 0, 0, 0, 0, 8, 8, 1, None) == 0


def test_path_selection():
    sel = gnt.gemm_nt_select_path
    al = 0x10000000
    # aligned, large -> tcgen05
    assert sel(al, al + 2 ** 26, al + 2 ** 27, 8192, 8192, 8192, 8192, 8192, 8192) == gnt.Path.TC05_PAIR
    assert sel(al, al, al, 128, 64, 64, 64, 64, 64) == gnt.Path.TC05
    assert sel(al, al, al, 128, 4096, 64, 64, 64, 4096) == gnt.Path.TC05
    # small M, long N -> swapped tcgen05 (skinny)
    assert sel(al, al, al, 64, 16384, 8192, 8192, 8192, 16384) == gnt.Path.SKINNY
    # ragged batched (K=1000: 2000-byte rows are 16-byte multiples) -> tcgen05
    assert sel(al, al, al, 3001, 2047, 1000, 1000, 1000, 2047, 3001000, 2047000, 3001 * 2047,
               16) == gnt.Path.TC05_PAIR
    # misaligned base, odd leading dimension or batch stride -> warp MMA kernel
    assert sel(al + 2, al, al, 256, 256, 256, 256, 256, 256) == gnt.Path.MMASYNC
    assert sel(al, al, al, 256, 256, 250, 250, 256, 256) == gnt.Path.MMASYNC
    assert sel(al, al, al, 256, 256, 256, 256, 256, 256, 65540, 65536, 65536, 2) == gnt.Path.MMASYNC


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(gnt, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        gnt.load(str(tmp_path / "nope.so"))


def test_dtype_validation(lib):
    """gemm_nt_batched_ex: unknown or unsupported element types, and an Out base
    not aligned to its own element size, are rejected on the host."""
    f = lib.gemm_nt_batched_ex
    D = gnt.DType
    base = (8, 8, 8, 8, 8, 8, 64, 64, 64, 1, 0, None)
    assert f(FAKE_A, FAKE_B, FAKE_O, D.F32, D.F32, *base) == gnt.Status.INVALID_VALUE  # fp32 inputs
    assert f(FAKE_A, FAKE_B, FAKE_O, 8, D.F32, *base) == gnt.Status.INVALID_VALUE
    assert f(FAKE_A, FAKE_B, FAKE_O, D.BF16, 9, *base) == gnt.Status.INVALID_VALUE
    assert f(FAKE_A, FAKE_B, FAKE_O + 1, D.F16, D.BF16, *base) == gnt.Status.INVALID_VALUE
    assert f(FAKE_A, FAKE_B, FAKE_O + 2, D.F16, D.F32, *base) == gnt.Status.INVALID_VALUE
    # a 16-bit Out of 8x8 ends 128 bytes after its base: ending inside B overlaps
    assert f(FAKE_A, FAKE_B, FAKE_B - 120, D.BF16, D.F16, *base) == gnt.Status.OVERLAP
    assert f(FAKE_A, FAKE_B, FAKE_O, D.BF16, D.F16, 0, 8, 8, 8, 8, 8, 64, 64, 64, 1, 0, None) == 0


def test_packed_validation(lib):
    """6- and 4-bit inputs: K-major only, whole-byte pitches and batch strides
    (fp4: even; fp6: multiples of 4 elements), and the overlap check counts
    their packed extent; all decided on the host."""
    f = lib.gemm_nt_batched_major
    D, Mj = gnt.DType, gnt.Major
    M, N, K = 8, 8, 256
    for ab, g in ((D.E2M1, 2), (D.E2M3, 4), (D.E3M2, 4)):
        ok = (FAKE_A, Mj.K, FAKE_B, Mj.K, FAKE_O, ab, D.F32, M, N, K, K, K, N, 0, 0, 0, 1, 0, None)
        assert f(*ok) not in (gnt.Status.INVALID_VALUE, gnt.Status.OVERLAP)
        # MN-major packed operands
        assert f(FAKE_A, Mj.MN, FAKE_B, Mj.K, FAKE_O, ab, D.F32, M, N, K, M + 8, K, N, 0, 0, 0, 1, 0,
                 None) == gnt.Status.INVALID_VALUE
        assert f(FAKE_A, Mj.K, FAKE_B, Mj.MN, FAKE_O, ab, D.F32, M, N, K, K, N + 8, N, 0, 0, 0, 1, 0,
                 None) == gnt.Status.INVALID_VALUE
        # a pitch that starts rows inside a byte (or a packing group)
        assert f(FAKE_A, Mj.K, FAKE_B, Mj.K, FAKE_O, ab, D.F32, M, N, K, K + g - 1, K, N, 0, 0, 0, 1, 0,
                 None) == gnt.Status.INVALID_VALUE
        assert f(FAKE_A, Mj.K, FAKE_B, Mj.K, FAKE_O, ab, D.F32, M, N, K, K, K + g - 1, N, 0, 0, 0, 1, 0,
                 None) == gnt.Status.INVALID_VALUE
        # a batch stride that does
        assert f(FAKE_A, Mj.K, FAKE_B, Mj.K, FAKE_O, ab, D.F32, M, N, K, K, K, N, M * K + g - 1, N * K,
                 M * N, 2, 0, None) == gnt.Status.INVALID_VALUE
        # A holds M*K*w/8 bytes: Out starting there does not overlap, 8 bytes before it does
        a_bytes = M * K * (4 if ab == D.E2M1 else 6) // 8
        assert f(FAKE_A, Mj.K, FAKE_B, Mj.K, FAKE_A + a_bytes, ab, D.F32, M, N, K, K, K, N, 0, 0, 0, 1, 0,
                 None) != gnt.Status.OVERLAP
        assert f(FAKE_A, Mj.K, FAKE_B, Mj.K, FAKE_A + a_bytes - 8, ab, D.F32, M, N, K, K, K, N, 0, 0, 0, 1, 0,
                 None) == gnt.Status.OVERLAP


def test_major_validation(lib):
    """gemm_nt_batched_major: an MN-major operand's pitch counts its stored rows'
    length (M or N), unknown majors are rejected, and the overlap check uses the
    stored extent."""
    f = lib.gemm_nt_batched_major
    D, Mj = gnt.DType, gnt.Major
    M, N, K = 16, 24, 8
    tail = (D.F16, D.F32, M, N, K)
    # A MN-major (stored K x M): lda must be >= M, not just >= K
    assert f(FAKE_A, Mj.MN, FAKE_B, Mj.K, FAKE_O, *tail, 8, 8, N, 0, 0, 0, 1, 0, None) == gnt.Status.INVALID_VALUE
    # B MN-major (stored K x N): ldb >= N
    assert f(FAKE_A, Mj.K, FAKE_B, Mj.MN, FAKE_O, *tail, 8, 16, N, 0, 0, 0, 1, 0, None) == gnt.Status.INVALID_VALUE
    assert f(FAKE_A, 2, FAKE_B, Mj.K, FAKE_O, *tail, 8, 8, N, 0, 0, 0, 1, 0, None) == gnt.Status.INVALID_VALUE
    assert f(FAKE_A, Mj.K, FAKE_B, -1, FAKE_O, *tail, 8, 8, N, 0, 0, 0, 1, 0, None) == gnt.Status.INVALID_VALUE
    # stored A is K x M = 8 x 16 fp16 = 256 bytes: Out 200 bytes after it overlaps
    assert f(FAKE_A, Mj.MN, FAKE_B, Mj.K, FAKE_A + 200, *tail, 16, 8, N, 0, 0, 0, 1, 0, None) == \
        gnt.Status.OVERLAP
    # an empty product returns before any pointer check
    assert f(FAKE_A, Mj.MN, FAKE_B, Mj.K, FAKE_A + 256, D.F16, D.F32, 0, N, K, 16, 8, N, 0, 0, 0, 1, 0,
             None) == 0


def test_mx_validation(lib):
    """Block-scaled entry: rejected on the host before any CUDA call."""
    D = gnt.DType
    f = lib.gemm_nt_mx
    tail = (64, 256, 256, 256, 256, 256, 0, 0, 0, 1, 0, None)  # M N K lda ldb ldo sA sB sO batch path stream
    SA, SB = FAKE_A + (1 << 20), FAKE_B + (1 << 20)
    assert f(FAKE_A, 0, FAKE_B, SB, FAKE_O, D.E4M3, D.F32, *tail) == gnt.Status.INVALID_VALUE  # null SA
    assert f(FAKE_A, SA, FAKE_B, 0, FAKE_O, D.E4M3, D.F32, *tail) == gnt.Status.INVALID_VALUE  # null SB
    assert f(FAKE_A, SA, FAKE_B, SB, FAKE_O, D.F16, D.F32, *tail) == gnt.Status.INVALID_VALUE  # 16-bit inputs
    assert f(FAKE_A, SA + 8, FAKE_B, SB, FAKE_O, D.E5M2, D.F32, *tail) == gnt.Status.INVALID_VALUE  # SA unaligned
    # Out on top of the scales of B
    assert f(FAKE_A, SA, FAKE_B, FAKE_O, FAKE_O, D.E4M3, D.F32, *tail) == gnt.Status.OVERLAP
    # empty problems launch nothing
    assert f(FAKE_A, 0, FAKE_B, 0, FAKE_O, D.E4M3, D.F32, 0, *tail[1:]) == gnt.Status.OK
    assert lib.gemm_nt_mx_scale_bytes(1, 1) == 512
    assert lib.gemm_nt_mx_scale_bytes(129, 257) == 2 * 3 * 512
    assert lib.gemm_nt_mx_scale_bytes(-1, 5) == -1
    p = lib.gemm_nt_mx_pack_scales
    assert p(0, 8, 0, FAKE_O, 10, 256, 1, None) == gnt.Status.INVALID_VALUE   # null plain
    assert p(FAKE_A, 7, 0, FAKE_O, 10, 256, 1, None) == gnt.Status.INVALID_VALUE  # ld < ceil(K/32)
    assert p(FAKE_A, 8, 8, FAKE_O, 10, 256, 2, None) == gnt.Status.INVALID_VALUE  # batch stride too small
    assert p(FAKE_A, 8, 0, FAKE_O, 0, 256, 1, None) == gnt.Status.OK          # nothing to pack


def test_no_alloc_validation(lib):
    """gemm_nt_f16_f32_batched_no_alloc checks its arguments before any CUDA
    call (no device here): bad arguments give their own status, not a CUDA
    failure, and empty products succeed without touching the device."""
    f = lib.gemm_nt_f16_f32_batched_no_alloc
    ok = (FAKE_A, FAKE_B, FAKE_O, 8, 8, 8, 8, 8, 8, 64, 64, 64, 1)
    assert f(*ok[:3], -1, *ok[4:], None) == gnt.Status.INVALID_VALUE              # negative M
    assert f(*ok[:6], 7, *ok[7:], None) == gnt.Status.INVALID_VALUE               # lda < K
    assert f(0, *ok[1:], None) == gnt.Status.INVALID_VALUE                        # null A
    assert f(FAKE_A, FAKE_B, FAKE_A + 64, *ok[3:], None) == gnt.Status.OVERLAP     # Out inside A
    assert f(*ok[:9], 64, 64, 63, 2, None) == gnt.Status.OVERLAP                 # batches of Out overlap
    assert f(*ok[:9], -64, 64, 64, 2, None) == gnt.Status.INVALID_VALUE          # negative stride
    assert f(*ok[:3], 0, *ok[4:], None) == gnt.Status.OK                           # M == 0
    assert f(*ok[:12], 0, None) == gnt.Status.OK                                  # batch == 0
