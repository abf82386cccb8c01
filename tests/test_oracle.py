"""The CPU oracle against its pins (no GPU)."""
import numpy as np
import pytest

import oracle
import oracle_pins
import workloads


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_golden_shapes_and_check(orc):
    """Shapes and tolerance printed with the two worked examples."""
    rows = [ln.split() for ln in open(_golden("worked_example_shapes.txt"))
            if ln.strip() and not ln.startswith("#")]
    assert [r[0] for r in rows] == ["warp_matrix", "blackwell_tcgen05"]
    rng = np.random.default_rng(21)
    for name, M, N, K, rtol, atol, _cols in rows:
        M, N, K, rtol, atol = int(M), int(N), int(K), float(rtol), float(atol)
        A = rng.standard_normal((M, K)).astype(np.float16)
        B = rng.standard_normal((N, K)).astype(np.float16)
        ref, _ = orc.gemm_nt(A, B)
        f32 = A.astype(np.float32) @ B.astype(np.float32).T
        np.testing.assert_allclose(ref, f32, rtol=rtol, atol=atol)


def test_workload_tile_matches_exact(orc):
    """The single-tile workload (A 128x64, B 64x64, uniform, seed 0) in full."""
    A, B = workloads.workload_inputs("tile_128x64x64")
    assert A.shape == (128, 64) and B.shape == (64, 64)
    oracle_pins.check_against_exact(orc, A, B)


def test_sampled_matches_full_on_ragged(orc):
    A, B = workloads.make_inputs(2, 37, 23, 45, "int4", seed=4)
    ref, absdot = orc.gemm_nt(A, B)
    rng = np.random.default_rng(0)
    b, i, j = rng.integers(0, 2, 64), rng.integers(0, 37, 64), rng.integers(0, 23, 64)
    s, sa = orc.gemm_nt_sampled(A, B, b, i, j)
    assert np.array_equal(s, ref[b, i, j]) and np.array_equal(sa, absdot[b, i, j])


def test_within_tolerance_predicate():
    ref = np.array([1.0, 0.0, 100.0])
    absdot = np.array([1.0, 0.0, 1000.0])
    assert oracle.within_tolerance([1.0 + 9e-4, 9e-7, 100.9], ref, absdot).all()
    assert not oracle.within_tolerance([1.0 + 1.2e-3, 0, 100], ref, absdot)[0]
    assert not oracle.within_tolerance([1.0, 2e-6, 100], ref, absdot)[1]


def _golden(name):
    import os
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", name)


def test_round_output_matches_library_casts():
    """round_output against torch's float32 -> float16 / bfloat16 casts (round
    to nearest even), hand-picked ties, and the float32 identity."""
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(5).standard_normal(1 << 15).astype(np.float32) * np.float32(3e3)
    x = np.concatenate([x, np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 2049.0, 2051.0, -2051.0, 0.0],
                                    dtype=np.float32)])
    t = torch.from_numpy(x)
    assert np.array_equal(oracle.round_output(x, "f16"), t.to(torch.float16).double().numpy())
    assert np.array_equal(oracle.round_output(x, "bf16"), t.to(torch.bfloat16).double().numpy())
    assert np.array_equal(oracle.round_output(x, "f32"), x.astype(np.float64))
    # ties go to even: 2049 -> 2048 and 2051 -> 2052 in float16; 1 + 2^-8 -> 1 in bfloat16
    assert oracle.round_output(np.array([2049.0, 2051.0]), "f16").tolist() == [2048.0, 2052.0]
    assert oracle.round_output(np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8]), "bf16").tolist() == \
        [1.0, 1 + 2.0 ** -6]
    with pytest.raises(ValueError):
        oracle.round_output(np.array([1 + 2.0 ** -40]), "f16")


def test_within_tolerance_widens_for_16_bit_outputs():
    ref = np.array([1000.0, 1000.0])
    absdot = np.array([0.0, 0.0])
    out = np.array([1000.0 + 0.48, 1000.0 + 3.8])
    assert oracle.within_tolerance(out, ref, absdot, "f16").tolist() == [True, False]
    assert oracle.within_tolerance(out, ref, absdot, "bf16").tolist() == [True, True]
    assert oracle.within_tolerance(out, ref, absdot, "f32").tolist() == [False, False]
