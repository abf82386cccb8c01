"""The warp-MMA register fragments on the GPU against the oracle's maps, which
are read from the printed layouts of "Warp Matrix Instructions" and pinned in
tests/test_fragments.py.  One warp runs the page's example (stage to shared
memory, ldmatrix.x4 / .x2, one mma.sync m16n8k16 with C = 0) and dumps its
registers lane by lane."""
import numpy as np
import pytest

import dense_fp16_tensor_gemm_gb300 as gnt
import oracle
from oracle import fragments as fr

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from dense_fp16_tensor_gemm_gb300 import _build
    _build.build()
    gnt.load()


def probe(A, B):
    import torch
    a = torch.from_numpy(np.ascontiguousarray(A)).cuda()
    b = torch.from_numpy(np.ascontiguousarray(B)).cuda()
    ar = torch.zeros((32, 4), dtype=torch.int32, device="cuda")
    br = torch.zeros((32, 2), dtype=torch.int32, device="cuda")
    dr = torch.zeros((32, 4), dtype=torch.float32, device="cuda")
    gnt.gemm_nt_probe_m16n8k16(a.data_ptr(), b.data_ptr(), ar.data_ptr(), br.data_ptr(),
                               dr.data_ptr(), torch.cuda.current_stream().cuda_stream)
    gnt.gemm_nt_check()
    return (ar.cpu().numpy().view(np.uint32), br.cpu().numpy().view(np.uint32),
            dr.cpu().numpy())


@pytest.mark.parametrize("seed", [0, 1])
def test_registers_match_fragment_maps(seed):
    rng = np.random.default_rng(seed)
    A = rng.standard_normal((16, 16)).astype(np.float16)
    B = rng.standard_normal((8, 16)).astype(np.float16)
    ar, br, dr = probe(A, B)
    want_ar, want_br = fr.fragments_from_matrices(A, B)
    assert np.array_equal(ar, want_ar), "A fragment (ldmatrix.x4) differs from the page's map"
    assert np.array_equal(br, want_br), "B fragment (ldmatrix.x2) differs from the page's map"
    _, want_dr = fr.warp_mma_via_fragments(A, B)
    ref, absdot = oracle.gemm_nt(A, B)
    # dr in lane/register order must hold the oracle's value at the D map's position
    for (lane, r), (row, col) in fr.d_mma_map().items():
        assert abs(dr[lane, r] - ref[row, col]) <= 1e-3 * absdot[row, col] + 1e-6


def test_coded_inputs_d_map():
    """A[i,0] = i, B[j,0] = 1 gives Out = i: dr[r] of lane l must read
    l//4 + 8*(r//2); A[i,0] = 1, B[j,0] = j gives 2*(l%4) + r%2."""
    A = np.zeros((16, 16), np.float16); B = np.zeros((8, 16), np.float16)
    A[:, 0] = np.arange(16); B[:, 0] = 1
    _, _, dr = probe(A, B)
    lanes = np.arange(32)[:, None]; regs = np.arange(4)[None, :]
    assert np.array_equal(dr, (lanes // 4 + 8 * (regs // 2)).astype(np.float32))
    A[:, 0] = 1; B[:, 0] = np.arange(8)
    _, _, dr = probe(A, B)
    assert np.array_equal(dr, (2 * (lanes % 4) + regs % 2).astype(np.float32))
