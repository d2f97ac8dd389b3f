"""GPU parity of the max-pooled block scores (needs a GB300).

The DSV pages ("Technische samenvatting" 2A/2B, Hindi summary 2A/2B) score a
group's proxy against key blocks with low-rank logits but leave the block
reduction open; dsv_predict_scores_max takes the tile maximum.  Gates, the
predictor's own: |dS| <= 1e-4 * max(|S_ref|, rms of the S_ref row) against the
fp64 oracle on the same bf16 inputs and fp32 W (the maximum moves by no more
than the largest logit error, and fp32 sums of r terms stay near 1e-6
relative); top-k lists of the GPU's max-pooled scores bit-exact against the
oracle fed those scores.  At the full latent16k size the oracle recomputes
sampled rows; the maximum is never below the tile mean at any size.
"""
import numpy as np
import pytest
import torch

import oracle
from dynamic_block_sparse_projection_gb300 import workloads as wl
from parity_util import SCORE_REL, SMALL, oracle_lists, score_err, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dynamic_block_sparse_projection_gb300 import binding
    return binding


@pytest.mark.parametrize("d,block,r,G", [(64, 64, 8, 18), (128, 128, 16, 18), (128, 64, 32, 18), (64, 128, 24, 18),
                                         (128, 128, 64, 18), (64, 64, 40, 17), (128, 64, 56, 21), (128, 128, 48, 5)])
def test_maxpool_all_shapes(dsv, d, block, r, G):
    """Every rank the kernels are built for and both block sizes; odd G at
    block 64 leaves the last 128-token tile half empty (rows past N are zero
    and their scores are not written), r = 56 and 64 take two query tiles per
    CTA instead of four, and the CTAs' step ranges cross from one query-tile
    group to the next mid-sweep."""
    B, H = 2, 2
    N = G * block
    g = torch.Generator(device="cuda").manual_seed(d + block + r)
    Q, K = (torch.randn(B, H, N, d, generator=g, device="cuda").to(torch.bfloat16) * 1.5 for _ in range(2))
    Wq, Wk = (torch.randn(H, d, r, generator=g, device="cuda") / d ** 0.5 for _ in range(2))
    S = dsv.predict_scores_max(Q, K, Wq, Wk, block)
    torch.cuda.synchronize()
    ref = oracle.predict_scores_max(to64(Q), to64(K), to64(Wq), to64(Wk), block)
    assert score_err(to64(S), ref) <= SCORE_REL
    # never below the tile mean of the same logits
    Sm = dsv.predict_scores(Q, K, Wq, Wk, block)
    assert torch.all(S >= Sm - 1e-4 * S.abs().amax())


@pytest.mark.parametrize("name", ["tiny", "latent16k_small", "long_small"])
def test_maxpool_workloads_and_topk(dsv, name):
    w = wl.WORKLOADS[name] if name in wl.WORKLOADS else SMALL[name]
    x = wl.make_inputs(w, device="cuda", with_dO=False)
    S = dsv.predict_scores_max(x.Q, x.K, x.Wq, x.Wk, w.block)
    torch.cuda.synchronize()
    ref = oracle.predict_scores_max(to64(x.Q), to64(x.K), to64(x.Wq), to64(x.Wk), w.block)
    assert score_err(to64(S), ref) <= SCORE_REL
    lists = dsv.topk_blocks(S, x.k_per_head, w.block, w.N, w.d)
    fp, fc, bp, bc = oracle_lists(to64(S), x.k_per_head, w.nb)
    got = [t.cpu().numpy().astype(np.int64) for t in lists]
    assert np.array_equal(got[0], fp) and np.array_equal(got[1][:len(fc)], fc)
    assert np.array_equal(got[2], bp) and np.array_equal(got[3][:len(bc)], bc)


def test_maxpool_full_size_sampled_rows(dsv):
    w = wl.WORKLOADS["latent16k"]
    x = wl.make_inputs(w, device="cuda", with_dO=False)
    S = dsv.predict_scores_max(x.Q, x.K, x.Wq, x.Wk, w.block)
    Sm = dsv.predict_scores(x.Q, x.K, x.Wq, x.Wk, w.block)
    torch.cuda.synchronize()
    rng = np.random.default_rng(77)
    rows = [(int(rng.integers(w.B)), int(rng.integers(w.H)), int(rng.integers(w.nb))) for _ in range(24)]
    rows += [(0, 0, 0), (w.B - 1, w.H - 1, w.nb - 1)]
    ref = oracle.predict_scores_max_rows(to64(x.Q), to64(x.K), to64(x.Wq), to64(x.Wk), w.block, rows)
    got = np.stack([to64(S[b, h, g]) for b, h, g in rows])
    assert score_err(got, ref) <= SCORE_REL
    assert torch.all(S >= Sm - 1e-4 * S.abs().amax())
    # repeatable bit for bit
    S2 = dsv.predict_scores_max(x.Q, x.K, x.Wq, x.Wk, w.block)
    assert torch.equal(S, S2)
