"""GPU parity of the 3D cube query grouping (needs a GB300): the token
permutation is bit-exact against the oracle's cube order (pure data
movement), and the hot path run on cube-ordered tokens matches the oracle run
on the oracle's permutation of the same inputs (DSV pages, "Technische
samenvatting" 2B and the Hindi summary 2B: queries grouped in 3D cubes)."""
import numpy as np
import pytest
import torch

import oracle
from dynamic_block_sparse_projection_gb300 import workloads as wl
from parity_util import (LSE_MAX_ABS, O_MAX_ABS, O_REL_L2, SMALL, max_abs_beyond_rounding, oracle_lists, rel_l2,
                         to64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dynamic_block_sparse_projection_gb300 import binding
    return binding


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy()


@pytest.mark.parametrize("B, H, grid, cube, d", [
    (1, 2, (4, 8, 8), (4, 4, 4), 128),
    (2, 3, (2, 16, 16), (2, 8, 8), 64),
    (1, 1, (2, 16, 32), (1, 8, 16), 128),
    (1, 2, (6, 10, 16), (1, 8, 8), 64),     # Hl % cy != 0: rejected
    (1, 1, (64, 90, 90), (2, 8, 8), 128),   # the long-video grid: rejected (90 % 8 != 0)
])
def test_cube_permute_bit_exact_and_round_trip(dsv, B, H, grid, cube, d):
    T, Hl, Wl = grid
    N = T * Hl * Wl
    g = torch.Generator(device="cuda").manual_seed(N + d)
    x = torch.randn(B, H, N, d, generator=g, device="cuda").to(torch.bfloat16)
    if Hl % cube[1] or Wl % cube[2] or T % cube[0]:
        with pytest.raises(dsv.DsvError):
            dsv.cube_permute(x, grid, cube)
        return
    y = dsv.cube_permute(x, grid, cube)
    z = dsv.cube_permute(y, grid, cube, inverse=True)
    torch.cuda.synchronize()
    perm = oracle.cube_order(*grid, *cube)
    assert np.array_equal(_bits(y), oracle.permute_tokens(_bits(x), perm))
    assert np.array_equal(_bits(z), _bits(x))


def test_hot_path_on_cube_order(dsv):
    """Permute Q, K, V into 2 x 8 x 8 cubes, run predictor, top-k and the
    forward on them, permute O back: equal (within the forward's tolerances)
    to the oracle's path on the oracle's permutation, with the GPU lists
    bit-exact against the oracle's top-k of the GPU scores."""
    w = SMALL["latent16k_small"]
    grid, cube = (w.T, w.Hl, w.Wl), (2, 8, 8)
    x = wl.make_inputs(w, device="cuda")
    Qc, Kc, Vc = (dsv.cube_permute(t, grid, cube) for t in (x.Q, x.K, x.V))
    S = dsv.predict_scores(Qc, Kc, x.Wq, x.Wk, w.block)
    fp, fc, bp, bc = dsv.topk_blocks(S, x.k_per_head, w.block, w.N, w.d)
    O, lse = dsv.sparse_attn_fwd(Qc, Kc, Vc, fp, fc, w.block)
    O_raster = dsv.cube_permute(O, grid, cube, inverse=True)
    torch.cuda.synchronize()
    assert dsv.device_error()[0] == 0

    perm = oracle.cube_order(*grid, *cube)
    Q, K, V = (oracle.permute_tokens(to64(t), perm) for t in (x.Q, x.K, x.V))
    S_gpu = to64(S)
    rfp, rfc, rbp, rbc = oracle_lists(S_gpu, x.k_per_head, w.nb)
    assert np.array_equal(fp.cpu().numpy(), rfp) and np.array_equal(fc.cpu().numpy(), rfc)
    assert np.array_equal(bp.cpu().numpy(), rbp) and np.array_equal(bc.cpu().numpy(), rbc)
    O_ref, L_ref = oracle.attn_fwd_groups(Q, K, V, rfp, rfc, w.block)
    O_ref_raster = oracle.permute_tokens(O_ref, perm, inverse=True)
    assert rel_l2(to64(O_raster), O_ref_raster) <= O_REL_L2
    assert max_abs_beyond_rounding(to64(O_raster), O_ref_raster) <= O_MAX_ABS
    assert np.max(np.abs(to64(lse) - L_ref)) <= LSE_MAX_ABS
