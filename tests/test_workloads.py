"""Seeded input generators (no GPU)."""
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
