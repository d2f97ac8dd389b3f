"""GPU parity of the mass-threshold selection (needs a GB300; DSV pages,
"Technische samenvatting" 2A and the Hindi summary 2A: the critical KV pairs
carry about 90 % of the attention score).

The oracle is fed the GPU's own fp32 scores.  The list size m of a row is an
integer decided by floating-point masses, which the kernel sums in exact
fixed point of fp32 exponentials and the oracle in fp64: m must lie between
the oracle's counts for tau - 1e-5 and tau + 1e-5 (equal to the exact count
unless the leading mass passes tau within that band), and then the list must
be the oracle's top m bit for bit; the transposed lists must be the oracle's
transpose.  The attention forward and backward then run on these
variable-length lists against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from dynamic_block_sparse_projection_gb300 import workloads as wl
from parity_util import (GRAD_REL_L2, O_MAX_ABS, O_REL_L2, SMALL, max_abs_beyond_rounding, rel_l2, to64)

pytestmark = pytest.mark.gpu

EPS = 1e-5


@pytest.fixture(scope="module")
def dsv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dynamic_block_sparse_projection_gb300 import binding
    return binding


def _check_lists(S64, fp, fc, bp, bc, tau, temp, kmin, kmax):
    B, H, G, nb = S64.shape
    fp, fc, bp, bc = (t.cpu().numpy().astype(np.int64) for t in (fp, fc, bp, bc))
    exact_rows = 0
    for r in range(B * H * G):
        b, rem = divmod(r, H * G)
        h, g = divmod(rem, G)
        row = S64[b, h, g]
        m = int(fp[r + 1] - fp[r])
        lo = oracle.mass_count_row(row, max(tau - EPS, 1e-12), temp, kmin, kmax)
        hi = oracle.mass_count_row(row, min(tau + EPS, 1.0), temp, kmin, kmax)
        assert kmin <= m <= kmax and lo <= m <= hi, (r, m, lo, hi)
        exact_rows += m == oracle.mass_count_row(row, tau, temp, kmin, kmax)
        assert np.array_equal(fc[fp[r]:fp[r + 1]], oracle.topk_row(row, m)), r
    tp, tc = oracle.transpose_lists(fp, fc, B, H, G, nb)
    assert np.array_equal(tp, bp) and np.array_equal(tc, bc[:len(tc)])
    return exact_rows / (B * H * G)


@pytest.mark.parametrize("name", ["tiny", "latent16k_small", "global_small", "long_small"])
@pytest.mark.parametrize("tau, kmin, kmax_frac", [(0.9, 1, 1.0), (0.5, 1, 1.0), (0.9, 2, 0.25), (1.0, 1, 1.0)])
def test_mass_lists_match_oracle(dsv, name, tau, kmin, kmax_frac):
    w = wl.WORKLOADS[name] if name in wl.WORKLOADS else SMALL[name]
    x = wl.make_inputs(w, device="cuda", with_dO=False)
    S = dsv.predict_scores(x.Q, x.K, x.Wq, x.Wk, w.block)
    kmax = max(kmin, int(round(kmax_frac * w.nb)))
    temp = 1.0 / np.sqrt(w.d)
    fp, fc, bp, bc = dsv.topk_mass_blocks(S, tau, w.block, w.N, w.d, temperature=temp, kmin=kmin, kmax=kmax)
    torch.cuda.synchronize()
    assert dsv.device_error()[0] == 0
    frac = _check_lists(to64(S), fp, fc, bp, bc, tau, temp, kmin, kmax)
    assert frac >= 0.99


def test_mass_lists_degenerate_rows(dsv):
    """Equal scores (m by division), a crowded value bucket (the radix levels),
    many ties, a large spread, tiny values and a non-finite score, on a
    hand-made score tensor (G = nb = 512)."""
    B, H, G = 1, 2, 512
    nb = G
    g = torch.Generator(device="cuda").manual_seed(5)
    S = torch.randn(B, H, G, nb, generator=g, device="cuda")
    ar = torch.arange(nb, device="cuda", dtype=torch.float32)
    S[0, 0, 0] = 0.75                                 # all equal
    S[0, 0, 1] = 1.0 + 1e-6 * ar                      # 511 scores in one value bucket beside an outlier
    S[0, 0, 1, 7] = -100.0
    S[0, 0, 2, :300] = 3.0                            # many ties far above the rest
    S[0, 0, 3] = torch.linspace(-40.0, 40.0, nb, device="cuda")         # large spread
    S[0, 0, 4, 17] = float("inf")                     # non-finite: m = kmax
    S[0, 1, 5] = -S[0, 1, 5].abs() * 1e-30            # tiny values
    temp, tau, kmax = 1.0, 0.9, 480
    fp, fc, bp, bc = dsv.topk_mass_blocks(S, tau, 64, nb * 64, 64, temperature=temp, kmin=1, kmax=kmax)
    torch.cuda.synchronize()
    assert dsv.device_error()[0] == 0
    fpn = fp.cpu().numpy()
    assert fpn[5] - fpn[4] == kmax
    assert fpn[1] - fpn[0] == int(np.ceil(0.9 * nb))
    _check_lists(to64(S), fp, fc, bp, bc, tau, temp, 1, kmax)


def test_attention_on_mass_lists(dsv):
    w = SMALL["latent16k_small"]
    x = wl.make_inputs(w, device="cuda")
    S = dsv.predict_scores(x.Q, x.K, x.Wq, x.Wk, w.block)
    fp, fc, bp, bc = dsv.topk_mass_blocks(S, 0.9, w.block, w.N, w.d)
    O, lse = dsv.sparse_attn_fwd(x.Q, x.K, x.V, fp, fc, w.block)
    dQ, dK, dV = dsv.sparse_attn_bwd(x.Q, x.K, x.V, O, x.dO, lse, fp, fc, bp, bc, w.block)
    torch.cuda.synchronize()
    assert dsv.device_error()[0] == 0
    fpn, fcn = fp.cpu().numpy().astype(np.int64), fc.cpu().numpy().astype(np.int64)
    lens = np.diff(fpn)
    assert lens.min() >= 1 and len(set(lens.tolist())) > 1          # variable row lengths
    Q, K, V, dO = (to64(t) for t in (x.Q, x.K, x.V, x.dO))
    O_ref, _ = oracle.attn_fwd_groups(Q, K, V, fpn, fcn, w.block)
    assert rel_l2(to64(O), O_ref) <= O_REL_L2
    assert max_abs_beyond_rounding(to64(O), O_ref) <= O_MAX_ABS
    rQ, rK, rV = oracle.attn_bwd_groups(Q, K, V, dO, fpn, fcn, w.block)
    for got, ref in ((dQ, rQ), (dK, rK), (dV, rV)):
        assert rel_l2(to64(got), ref) <= GRAD_REL_L2
