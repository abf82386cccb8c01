"""Seeded synthetic inputs for the fp16 product Out = A @ B.T.

This module holds the five workloads and their input recipe, and nothing of
the product's arithmetic: it only draws random numbers and rounds them to fp16.
Both sides of every parity check (the CPU oracle and the CUDA library) receive
the arrays made here, so they see identical bits.

Recipe (one ``numpy.random.default_rng(seed)`` stream per workload):
  * A is drawn first (batch-major, then row-major), then B, from the same stream;
  * uniform[-1,1]  -> ``rng.uniform(-1.0, 1.0)`` in float64;
  * normal(0, s)   -> ``s * rng.standard_normal()`` in float64;
  * integers [-4,4]-> ``rng.integers(-4, 5, dtype=int8)`` (inclusive bounds);
  * every value is then rounded once to fp16 with round-to-nearest-even
    (numpy's float64 -> float16 cast); values stay far inside fp16's range, and
    normal(0, 0.02) yields some fp16 subnormals, which are kept.
Float draws are made in chunks of 2**24 values; the stream is sequential, so
the chunking does not change the values.

bfloat16 inputs (``dtype="bf16"``) come from the same draws: each float64 value
is cast to float32 (numpy, round to nearest even) and the float32 is rounded to
its upper 16 bits, again to nearest with ties to even.  They are returned as
uint16 bit patterns (numpy has no bfloat16 type).

8-bit float inputs (``dtype="e4m3"`` or ``"e5m2"``) also come from the same
draws: float64 -> float32 (numpy), then torch's float32 -> float8 cast (round
to nearest even; every drawn value lies inside both formats' ranges).  They are
returned as uint8 bit patterns.
"""
from dataclasses import dataclass

import numpy as np

_CHUNK = 1 << 24


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    M: int
    N: int
    K: int
    dist: str          # "uniform", "normal" or "int4"
    sigma: float       # for "normal"
    seed: int
    description: str

    @property
    def flops(self) -> float:
        return 2.0 * self.batch * self.M * self.N * self.K

    @property
    def bytes(self) -> float:
        """Algorithmic bytes: read A and B once (fp16), write Out once (fp32)."""
        return float(self.batch) * (2 * self.M * self.K + 2 * self.N * self.K + 4 * self.M * self.N)


WORKLOADS = {
    "tile_128x64x64": Workload(
        "tile_128x64x64", 1, 128, 64, 64, "uniform", 0.0, 0,
        "A (128,64), B (64,64), uniform[-1,1], seed 0: one CTA tile"),
    "square_4096": Workload(
        "square_4096", 1, 4096, 4096, 4096, "uniform", 0.0, 1,
        "M=N=K=4096, uniform[-1,1], seed 1"),
    "square_8192": Workload(
        "square_8192", 1, 8192, 8192, 8192, "normal", 1.0, 2,
        "M=N=K=8192, normal(0,1), seed 2 (compute-bound headline)"),
    "skinny_64x16384x8192": Workload(
        "skinny_64x16384x8192", 1, 64, 16384, 8192, "normal", 0.02, 3,
        "M=64, N=16384, K=8192, normal(0,0.02), seed 3 (memory-bound)"),
    "ragged_batch16_3001x2047x1000": Workload(
        "ragged_batch16_3001x2047x1000", 16, 3001, 2047, 1000, "int4", 0.0, 4,
        "batch 16 of M=3001, N=2047, K=1000, integers in [-4,4], seed 4 (exact)"),
}


def _draw(rng, n, dist, sigma):
    out = np.empty(n, dtype=np.float16)
    if dist == "int4":
        out[:] = rng.integers(-4, 5, size=n, dtype=np.int8)
        return out
    for s in range(0, n, _CHUNK):
        m = min(_CHUNK, n - s)
        if dist == "uniform":
            out[s:s + m] = rng.uniform(-1.0, 1.0, size=m)
        elif dist == "normal":
            out[s:s + m] = sigma * rng.standard_normal(size=m)
        else:
            raise ValueError("unknown distribution %r" % dist)
    return out


def float32_to_bf16_bits(x):
    """Round float32 values to bfloat16, nearest with ties to even, returning
    the uint16 bit patterns.  Inputs here are finite, so no NaN case is needed."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


def _draw_bf16(rng, n, dist, sigma):
    out = np.empty(n, dtype=np.uint16)
    if dist == "int4":
        out[:] = float32_to_bf16_bits(rng.integers(-4, 5, size=n, dtype=np.int8).astype(np.float32))
        return out
    for s in range(0, n, _CHUNK):
        m = min(_CHUNK, n - s)
        if dist == "uniform":
            v = rng.uniform(-1.0, 1.0, size=m)
        elif dist == "normal":
            v = sigma * rng.standard_normal(size=m)
        else:
            raise ValueError("unknown distribution %r" % dist)
        out[s:s + m] = float32_to_bf16_bits(v.astype(np.float32))
    return out


def _draw_f8(dtype):
    import torch
    tt = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}[dtype]

    def draw(rng, n, dist, sigma):
        out = np.empty(n, dtype=np.uint8)
        if dist == "int4":
            v = rng.integers(-4, 5, size=n, dtype=np.int8).astype(np.float32)
            out[:] = torch.from_numpy(v).to(tt).view(torch.uint8).numpy()
            return out
        for s in range(0, n, _CHUNK):
            m = min(_CHUNK, n - s)
            if dist == "uniform":
                v = rng.uniform(-1.0, 1.0, size=m)
            elif dist == "normal":
                v = sigma * rng.standard_normal(size=m)
            else:
                raise ValueError("unknown distribution %r" % dist)
            out[s:s + m] = torch.from_numpy(v.astype(np.float32)).to(tt).view(torch.uint8).numpy()
        return out
    return draw


# 6- and 4-bit floats, one per byte in its low bits: (exponent bits, fraction
# bits, bias).  Inputs are drawn as values and rounded to the nearest value of
# the format (ties to the even code), which needs the format's value grid.
F6F4 = {"e2m3": (2, 3, 1), "e3m2": (3, 2, 3), "e2m1": (2, 1, 1)}


def _f6f4_grid(dtype):
    """(values, codes) of the non-negative codes of a 6- or 4-bit format,
    ascending."""
    e, m, b = F6F4[dtype]
    vals, codes = [], []
    for expo in range(2 ** e):
        for frac in range(2 ** m):
            vals.append(frac / 2 ** m * 2.0 ** (1 - b) if expo == 0 else (1 + frac / 2 ** m) * 2.0 ** (expo - b))
            codes.append((expo << m) | frac)
    return np.array(vals), np.array(codes, dtype=np.uint8)


def _draw_f6f4(dtype):
    vals, codes = _f6f4_grid(dtype)
    e, m, b = F6F4[dtype]
    sign_bit = np.uint8(1 << (e + m))

    def quantize(v):
        a = np.minimum(np.abs(v), vals[-1])
        hi = np.clip(np.searchsorted(vals, a), 1, len(vals) - 1)
        lo = hi - 1
        d_lo, d_hi = a - vals[lo], vals[hi] - a
        pick = np.where((d_hi < d_lo) | ((d_hi == d_lo) & (codes[hi] % 2 == 0)), hi, lo)
        return codes[pick] | np.where(v < 0, sign_bit, np.uint8(0))

    def draw(rng, n, dist, sigma):
        out = np.empty(n, dtype=np.uint8)
        if dist == "int4":
            out[:] = quantize(rng.integers(-4, 5, size=n, dtype=np.int8).astype(np.float64))
            return out
        for s in range(0, n, _CHUNK):
            m_ = min(_CHUNK, n - s)
            if dist == "uniform":
                v = rng.uniform(-1.0, 1.0, size=m_)
            elif dist == "normal":
                v = sigma * rng.standard_normal(size=m_)
            else:
                raise ValueError("unknown distribution %r" % dist)
            out[s:s + m_] = quantize(v)
        return out
    return draw


def pack_subbyte(codes, dtype):
    """Codes of a 6- or 4-bit format (uint8, one per element, (..., K) with K a
    multiple of 4 or 2) -> the packed storage along the last axis: element k
    at bits [b*k, b*k + b) of the row's little-endian bit string (b = 6 or 4)."""
    e, m, _ = F6F4[dtype]
    b = 1 + e + m
    c = np.asarray(codes, dtype=np.uint8) & np.uint8((1 << b) - 1)
    K = c.shape[-1]
    if b == 4:
        if K % 2:
            raise ValueError("fp4 rows need an even number of elements")
        return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)
    if K % 4:
        raise ValueError("fp6 rows need a multiple of 4 elements")
    g = c.reshape(c.shape[:-1] + (K // 4, 4)).astype(np.uint32)
    word = g[..., 0] | (g[..., 1] << 6) | (g[..., 2] << 12) | (g[..., 3] << 18)
    out = np.stack([word & 0xff, (word >> 8) & 0xff, (word >> 16) & 0xff], axis=-1).astype(np.uint8)
    return out.reshape(c.shape[:-1] + (K // 4 * 3,))


def make_inputs(batch, M, N, K, dist="uniform", sigma=1.0, seed=0, dtype="f16"):
    """Return (A, B) of shape (batch,M,K), (batch,N,K) (or (M,K), (N,K) when
    batch == 0 is passed to mean "unbatched"): float16 arrays for dtype "f16",
    uint16 bfloat16 bit patterns for dtype "bf16", uint8 patterns for "e4m3"
    and "e5m2", and for the 6- and 4-bit floats "e2m3", "e3m2", "e2m1" (values
    rounded to the nearest code, one code per byte; pack_subbyte gives the
    packed storage the library takes)."""
    rng = np.random.default_rng(seed)
    nb = max(batch, 1)
    if dtype in ("f16", "bf16"):
        draw = {"f16": _draw, "bf16": _draw_bf16}[dtype]
    else:
        draw = _draw_f6f4(dtype) if dtype in F6F4 else _draw_f8(dtype)
    A = draw(rng, nb * M * K, dist, sigma).reshape(nb, M, K)
    B = draw(rng, nb * N * K, dist, sigma).reshape(nb, N, K)
    if batch == 0:
        return A[0], B[0]
    return A, B


def workload_inputs(name, dtype="f16"):
    """Inputs of a named workload: 2-D for batch 1, 3-D otherwise."""
    w = WORKLOADS[name]
    return make_inputs(0 if w.batch == 1 else w.batch, w.M, w.N, w.K, w.dist, w.sigma, w.seed, dtype)


def workload_mx_scales(name):
    """Seeded block scales of a named workload for the block-scaled product:
    E8M0 bytes uniform in 120..134 (2^-7..2^7), one per 32 K elements of each
    row, (rows, ceil(K/32)) for batch 1 else (batch, rows, ceil(K/32)); A's,
    then B's."""
    w = WORKLOADS[name]
    rng = np.random.default_rng(w.seed + 7)
    kb = (w.K + 31) // 32
    sa = rng.integers(120, 135, size=(w.batch, w.M, kb)).astype(np.uint8)
    sb = rng.integers(120, 135, size=(w.batch, w.N, kb)).astype(np.uint8)
    if w.batch == 1:
        sa, sb = sa[0], sb[0]
    return sa, sb
