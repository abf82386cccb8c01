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
