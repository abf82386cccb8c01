"""The oracle's register-fragment maps (oracle/fragments.py) against the pages'
independent statements of them (no GPU).

"Warp Matrix Instructions", "From Shared Memory to a Matrix Product" states the
maps three ways: the ``S[...]`` layouts, the explicit store loop and the lane-0
example.  "copy -> ldstmatrix", "Algorithm" step 2, states the ldmatrix lane rule
(lane i holds row i//4 and column pair i%4).  Each is checked against the others.
"""
import os

import numpy as np
import pytest

import oracle
from oracle import fragments as fr


def _golden_lane0():
    path = os.path.join(os.path.dirname(__file__), "golden", "warp_example_lane0_d.txt")
    return [tuple(int(x) for x in ln.split()) for ln in open(path)
            if ln.strip() and not ln.startswith("#")]


def test_register_counts():
    # ar: four words, br: two words, dr: four floats per lane (the page's table)
    a, b, d = fr.a_load_map(), fr.b_load_map(), fr.d_mma_map()
    assert max(r for _, r in a) + 1 == 4 and max(r for _, r in b) + 1 == 2
    assert max(r for _, r in d) + 1 == 4
    assert {l for l, _ in a} == {l for l, _ in b} == {l for l, _ in d} == set(range(32))


@pytest.mark.parametrize("mapping,cells", [
    (fr.a_load_map, 16 * 8), (fr.b_load_map, 8 * 8), (fr.a_mma_map, 16 * 8),
    (fr.b_mma_map, 8 * 8), (fr.d_mma_map, 16 * 8)])
def test_maps_are_bijections(mapping, cells):
    m = mapping()
    assert len(m) == cells and len(set(m.values())) == cells


def test_d_layout_matches_store_loop_and_lane0():
    d = fr.d_mma_map()
    for (lane, r), (row, col) in d.items():
        assert fr.store_loop_coords(lane, r) == (row, col)
    for lane, r, row, col in _golden_lane0():
        assert d[(lane, r)] == (row, col)


def test_ldmatrix_lane_rule():
    """Within every 8x8 matrix, lane i holds row i//4 and 32-bit column pair i%4."""
    for (lane, reg), (row, word) in fr.a_load_map().items():
        assert row % 8 == lane // 4 and word % 4 == lane % 4
    for (lane, reg), (row, word) in fr.b_load_map().items():
        assert row == lane // 4 and word % 4 == lane % 4


def test_mma_views_read_the_loaded_registers():
    """Both instructions use the same fragments without moving values between
    lanes: the load and MMA maps agree register for register."""
    assert fr.a_load_map() == fr.a_mma_map()
    assert fr.b_load_map() == fr.b_mma_map()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_fragment_product_equals_oracle(seed):
    rng = np.random.default_rng(seed)
    A = rng.standard_normal((16, 16)).astype(np.float16)
    B = rng.standard_normal((8, 16)).astype(np.float16)
    out, _ = fr.warp_mma_via_fragments(A, B)
    ref, absdot = oracle.gemm_nt(A, B)
    assert np.all(np.abs(out - ref) <= 1e-13 * absdot)


def test_planted_layout_mistake_is_caught(monkeypatch):
    """Swapping the lane strides of A's load layout scrambles the product."""
    monkeypatch.setattr(fr, "A_LOAD", [(4, 1, fr.REG), (8, 1, fr.LANE), (4, 8, fr.LANE)])
    rng = np.random.default_rng(0)
    A = rng.standard_normal((16, 16)).astype(np.float16)
    B = rng.standard_normal((8, 16)).astype(np.float16)
    out, _ = fr.warp_mma_via_fragments(A, B)
    ref, _ = oracle.gemm_nt(A, B)
    assert not np.allclose(out, ref)
