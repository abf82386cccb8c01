"""Seeded input generators (no GPU)."""
import pytest
import numpy as np

import workloads


def test_deterministic_and_seed_dependent():
    a1, b1 = workloads.make_inputs(0, 50, 40, 30, "normal", 1.0, seed=2)
    a2, b2 = workloads.make_inputs(0, 50, 40, 30, "normal", 1.0, seed=2)
    a3, _ = workloads.make_inputs(0, 50, 40, 30, "normal", 1.0, seed=3)
    assert a1.dtype == np.float16 and b1.dtype == np.float16
    assert np.array_equal(a1.view(np.uint16), a2.view(np.uint16))
    assert np.array_equal(b1.view(np.uint16), b2.view(np.uint16))
    assert not np.array_equal(a1, a3)


def test_distributions():
    a, b = workloads.make_inputs(0, 200, 100, 256, "uniform", seed=1)
    assert a.min() >= -1 and a.max() <= 1 and abs(float(a.astype(np.float64).mean())) < 0.02
    a, _ = workloads.make_inputs(0, 256, 8, 256, "normal", 0.02, seed=3)
    assert abs(float(a.astype(np.float64).std()) - 0.02) < 1e-3
    a, b = workloads.make_inputs(3, 30, 20, 50, "int4", seed=4)
    assert a.shape == (3, 30, 50) and b.shape == (3, 20, 50)
    vals = set(np.unique(np.concatenate([a.ravel(), b.ravel()])).tolist())
    assert vals == set(float(v) for v in range(-4, 5))


def test_chunking_does_not_change_values(monkeypatch):
    full = workloads.make_inputs(0, 64, 8, 100, "normal", 1.0, seed=7)
    monkeypatch.setattr(workloads, "_CHUNK", 37)
    chunked = workloads.make_inputs(0, 64, 8, 100, "normal", 1.0, seed=7)
    assert all(np.array_equal(x, y) for x, y in zip(full, chunked))


def test_workload_table():
    w = workloads.WORKLOADS
    assert (w["square_8192"].M, w["square_8192"].K) == (8192, 8192)
    assert w["skinny_64x16384x8192"].bytes == 2 * 64 * 8192 + 2 * 16384 * 8192 + 4 * 64 * 16384
    r = w["ragged_batch16_3001x2047x1000"]
    assert (r.batch, r.M, r.N, r.K, r.dist) == (16, 3001, 2047, 1000, "int4")


def test_bf16_rounding_is_nearest_even():
    """Hand cases (ties go to the even pattern) and agreement with torch's own
    float32 -> bfloat16 cast on many random values."""
    torch = __import__("pytest").importorskip("torch")
    f = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 1.0 + 2.0 ** -7,
                  2.0 ** -130, 0.0, -0.0], dtype=np.float32)
    got = workloads.float32_to_bf16_bits(f)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7 -> 1 (even); 1 + 3*2^-8 -> 1 + 2^-6;
    # 2^-130 is the subnormal 8 * 2^-133
    assert got.tolist() == [0x3F80, 0x3F80, 0x3F82, 0xBF80, 0x3F81, 0x0008, 0x0000, 0x8000]
    x = np.random.default_rng(0).standard_normal(1 << 16).astype(np.float32) * np.float32(1e3)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(workloads.float32_to_bf16_bits(x), want)


def test_bf16_inputs_follow_the_same_draws():
    a16, b16 = workloads.make_inputs(2, 30, 20, 50, "int4", seed=4)
    a, b = workloads.make_inputs(2, 30, 20, 50, "int4", seed=4, dtype="bf16")
    assert a.dtype == np.uint16 and a.shape == (2, 30, 50)
    dec = lambda x: (x.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(dec(a), a16.astype(np.float32)) and np.array_equal(dec(b), b16.astype(np.float32))
    a, _ = workloads.make_inputs(0, 64, 8, 100, "normal", 0.02, seed=7, dtype="bf16")
    assert a.shape == (64, 100) and abs(float(dec(a).std()) - 0.02) < 2e-3


def test_f8_inputs_follow_the_same_draws():
    torch = __import__("pytest").importorskip("torch")
    for dtype, tt in (("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)):
        a16, _ = workloads.make_inputs(0, 20, 10, 40, "int4", seed=4)
        a, b = workloads.make_inputs(0, 20, 10, 40, "int4", seed=4, dtype=dtype)
        assert a.dtype == np.uint8 and a.shape == (20, 40) and b.shape == (10, 40)
        dec = torch.from_numpy(a.copy()).view(tt).to(torch.float64).numpy()
        assert np.array_equal(dec, a16.astype(np.float64))
        x, _ = workloads.make_inputs(0, 64, 8, 256, "normal", 1.0, seed=5, dtype=dtype)
        v = torch.from_numpy(x.copy()).view(tt).to(torch.float64).numpy()
        assert np.isfinite(v).all() and abs(float(v.std()) - 1.0) < 0.1


def _unpack_bits(packed, bits, K):
    """Independent reading of the packed rows: the row as one little-endian
    bit string (numpy's unpackbits, bit order little), element k = bits
    [bits*k, bits*k + bits)."""
    flat = np.unpackbits(np.asarray(packed, dtype=np.uint8), axis=-1, bitorder="little")
    flat = flat[..., : bits * K].reshape(packed.shape[:-1] + (K, bits))
    return (flat * (1 << np.arange(bits))).sum(axis=-1).astype(np.uint8)


def test_subbyte_packing_rule_and_round_trip():
    """pack_subbyte: hand-worked bytes, and every code at every position read
    back through an independent bit-string decoding."""
    assert workloads.pack_subbyte(np.array([[1, 2, 3, 4]], np.uint8), "e2m3").tolist() == [[0x81, 0x30, 0x10]]
    assert workloads.pack_subbyte(np.array([[1, 2, 15, 7]], np.uint8), "e2m1").tolist() == [[0x21, 0x7F]]
    rng = np.random.default_rng(0)
    for dtype, bits in (("e2m1", 4), ("e2m3", 6), ("e3m2", 6)):
        codes = rng.integers(0, 1 << bits, size=(3, 5, 64)).astype(np.uint8)
        packed = workloads.pack_subbyte(codes, dtype)
        assert packed.shape == (3, 5, 64 * bits // 8)
        assert np.array_equal(_unpack_bits(packed, bits, 64), codes)
    with pytest.raises(ValueError):
        workloads.pack_subbyte(np.zeros((2, 3), np.uint8), "e2m1")
    with pytest.raises(ValueError):
        workloads.pack_subbyte(np.zeros((2, 6), np.uint8), "e3m2")


def test_subbyte_draws_are_codes_of_the_format():
    """The 6- and 4-bit draws: codes within the format's width, the sign bit
    set exactly for negative draws (a zero code may carry either sign), and
    every magnitude code reachable for normal(0,1) over enough draws."""
    for dtype, bits in (("e2m1", 4), ("e2m3", 6), ("e3m2", 6)):
        A, B = workloads.make_inputs(0, 64, 64, 256, "normal", 1.0, seed=11, dtype=dtype)
        assert A.dtype == np.uint8 and int(A.max()) < (1 << bits)
        mags = np.unique(np.concatenate([A.ravel(), B.ravel()]) & ((1 << (bits - 1)) - 1))
        assert len(mags) >= (1 << (bits - 1)) // 2
    # integers 0..4 are exact in E2M1: magnitude codes 0, 2, 4, 5, 6 (0, 1, 2, 3, 4)
    I, _ = workloads.make_inputs(0, 8, 8, 128, "int4", seed=1, dtype="e2m1")
    assert set(np.unique(I & 7).tolist()) == {0, 2, 4, 5, 6}


def test_mx_scale_recipe():
    sa, sb = workloads.workload_mx_scales("square_4096")
    assert sa.shape == (4096, 128) and sb.shape == (4096, 128)
    assert sa.min() >= 120 and sa.max() <= 134
    sa2, _ = workloads.workload_mx_scales("square_4096")
    assert np.array_equal(sa, sa2)
    sr, _ = workloads.workload_mx_scales("ragged_batch16_3001x2047x1000")
    assert sr.shape == (16, 3001, 32)
