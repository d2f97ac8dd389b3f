"""GPU parity of the predictor, top-k and sparse attention forward (needs a GB300).

Every comparison is against the fp64 oracle on the same seeded inputs:
  * predictor scores: |dS| <= 1e-4 * max(|S_ref|, row rms);
  * top-k lists: bit-exact against the oracle's top-k of the GPU's own scores
    (the selection is an integer decision taken on fp32 keys on both sides);
  * attention forward: O rel-L2 <= 1e-2 and max-abs <= 2e-2 beyond the
    bf16 output's own rounding (half a bf16 ulp of the oracle value), against
    the oracle run on lists the oracle computed itself.
"""
import numpy as np
import pytest
import torch

import oracle
from dynamic_block_sparse_projection_gb300 import workloads as wl
from parity_util import (LSE_MAX_ABS, O_MAX_ABS, O_REL_L2, SCORE_REL, SMALL, csr_to_device,
                         max_abs_beyond_rounding, oracle_lists, random_lists, rel_l2, score_err, to64)

pytestmark = pytest.mark.gpu

CASES = ["tiny"] + list(SMALL)


def _workload(name):
    return wl.WORKLOADS[name] if name in wl.WORKLOADS else SMALL[name]


@pytest.fixture(scope="module")
def dsv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dynamic_block_sparse_projection_gb300 import binding
    return binding


@pytest.mark.parametrize("name", CASES)
def test_predictor_and_topk_match_oracle(dsv, name):
    w = _workload(name)
    x = wl.make_inputs(w, device="cuda")
    S = dsv.predict_scores(x.Q, x.K, x.Wq, x.Wk, w.block)
    fp, fc, bp, bc = dsv.topk_blocks(S, x.k_per_head, w.block, w.N, w.d)
    torch.cuda.synchronize()
    assert dsv.device_error()[0] == 0
    S_ref = oracle.predict_scores(to64(x.Q), to64(x.K), to64(x.Wq), to64(x.Wk), w.block)
    S_gpu = to64(S)
    err = score_err(S_gpu, S_ref)
    assert err <= SCORE_REL, f"score error {err:.3e}"
    rfp, rfc, rbp, rbc = oracle_lists(S_gpu, x.k_per_head, w.nb)
    assert np.array_equal(fp.cpu().numpy(), rfp)
    assert np.array_equal(fc.cpu().numpy(), rfc)
    assert np.array_equal(bp.cpu().numpy(), rbp)
    assert np.array_equal(bc.cpu().numpy(), rbc)


@pytest.mark.parametrize("name", CASES)
def test_forward_matches_oracle(dsv, name):
    w = _workload(name)
    x = wl.make_inputs(w, device="cuda")
    Q, K, V = (to64(t) for t in (x.Q, x.K, x.V))
    S_ref = oracle.predict_scores(Q, K, to64(x.Wq), to64(x.Wk), w.block)
    rfp, rfc, _, _ = oracle_lists(S_ref, x.k_per_head, w.nb)
    fp, fc = csr_to_device((rfp, rfc), "cuda")
    O, lse = dsv.sparse_attn_fwd(x.Q, x.K, x.V, fp, fc, w.block)
    torch.cuda.synchronize()
    assert dsv.device_error()[0] == 0
    O_ref, L_ref = oracle.attn_fwd_groups(Q, K, V, rfp, rfc, w.block)
    O_gpu = to64(O)
    assert rel_l2(O_gpu, O_ref) <= O_REL_L2
    assert max_abs_beyond_rounding(O_gpu, O_ref) <= O_MAX_ABS
    assert np.max(np.abs(to64(lse) - L_ref)) <= LSE_MAX_ABS


@pytest.mark.parametrize("block,d", [(64, 64), (64, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("k", [1, 3, "all"])
def test_forward_all_tile_shapes(dsv, block, d, k):
    rng = np.random.default_rng(block * 1000 + d + (0 if k == "all" else k))
    B, H, G = 1, 2, 5
    N = G * block
    kk = G if k == "all" else k
    g = torch.Generator(device="cuda").manual_seed(7)
    Qb, Kb, Vb = (torch.randn(B, H, N, d, generator=g, device="cuda").to(torch.bfloat16) * 2 for _ in range(3))
    fp_, fc_, _, _ = random_lists(rng, B, H, G, [kk, kk])
    fp, fc = csr_to_device((fp_, fc_), "cuda")
    O, lse = dsv.sparse_attn_fwd(Qb, Kb, Vb, fp, fc, block)
    torch.cuda.synchronize()
    O_ref, L_ref = oracle.attn_fwd_groups(to64(Qb), to64(Kb), to64(Vb), fp_, fc_, block)
    assert rel_l2(to64(O), O_ref) <= O_REL_L2
    assert max_abs_beyond_rounding(to64(O), O_ref) <= O_MAX_ABS
    assert np.max(np.abs(to64(lse) - L_ref)) <= LSE_MAX_ABS


def test_forward_dense_equals_masked_dense(dsv):
    """k = nb: the sparse kernel is dense attention (the oracle's literal masked form)."""
    B, H, N, d, block = 1, 2, 512, 128, 128
    G = N // block
    g = torch.Generator(device="cuda").manual_seed(3)
    Qb, Kb, Vb = (torch.randn(B, H, N, d, generator=g, device="cuda").to(torch.bfloat16) for _ in range(3))
    fp_ = np.arange(0, B * H * G * G + 1, G)
    fc_ = np.tile(np.arange(G), B * H * G)
    fp, fc = csr_to_device((fp_, fc_), "cuda")
    O, _ = dsv.sparse_attn_fwd(Qb, Kb, Vb, fp, fc, block)
    mask = np.ones((B, H, G, G), bool)
    O_ref, _ = oracle.attn_fwd_masked(to64(Qb), to64(Kb), to64(Vb), mask, block)
    assert rel_l2(to64(O), O_ref) <= O_REL_L2


def test_forward_later_blocks_far_above_the_first(dsv):
    """The forward's reference maximum is each row's first block's; a later
    block whose values of P would pass 2^64 must take its own maximum and
    rescale O.  Key blocks 1, 2, 3 are scaled by 3, 12 and 40 against 0.1 for
    block 0, so the last blocks' exponents run far past 64 (and past the fp32
    range) above the first block's maximum; the result must still be the
    oracle's."""
    B, H, N, d, block = 1, 2, 256, 64, 64
    G = N // block
    g = torch.Generator(device="cuda").manual_seed(11)
    Qb = (torch.randn(B, H, N, d, generator=g, device="cuda") * 4).to(torch.bfloat16)
    Kf = torch.randn(B, H, N, d, generator=g, device="cuda")
    for j, f in enumerate((0.1, 3.0, 12.0, 40.0)):
        Kf[:, :, j * block:(j + 1) * block] *= f
    Kb = Kf.to(torch.bfloat16)
    Vb = torch.randn(B, H, N, d, generator=g, device="cuda").to(torch.bfloat16)
    fp_ = np.arange(0, B * H * G * G + 1, G)
    fc_ = np.tile(np.arange(G), B * H * G)                # every row: blocks 0, 1, 2, 3 in this order
    fp, fc = csr_to_device((fp_, fc_), "cuda")
    O, lse = dsv.sparse_attn_fwd(Qb, Kb, Vb, fp, fc, block)
    torch.cuda.synchronize()
    assert dsv.device_error()[0] == 0
    O_ref, L_ref = oracle.attn_fwd_groups(to64(Qb), to64(Kb), to64(Vb), fp_, fc_, block)
    assert np.all(np.isfinite(to64(O))) and np.all(np.isfinite(to64(lse)))
    assert rel_l2(to64(O), O_ref) <= O_REL_L2
    assert max_abs_beyond_rounding(to64(O), O_ref) <= O_MAX_ABS
    assert np.max(np.abs(to64(lse) - L_ref)) <= LSE_MAX_ABS


def test_forward_empty_list_and_custom_scale(dsv):
    B, H, N, d, block = 1, 1, 256, 64, 64
    g = torch.Generator(device="cuda").manual_seed(5)
    Qb, Kb, Vb = (torch.randn(B, H, N, d, generator=g, device="cuda").to(torch.bfloat16) for _ in range(3))
    fp_ = np.array([0, 2, 2, 3, 4])        # group 1 has an empty list
    fc_ = np.array([1, 3, 0, 2])
    fp, fc = csr_to_device((fp_, fc_), "cuda")
    O, lse = dsv.sparse_attn_fwd(Qb, Kb, Vb, fp, fc, block, softmax_scale=0.2)
    torch.cuda.synchronize()
    O, lse = to64(O), to64(lse)
    assert np.all(O[0, 0, 64:128] == 0) and np.all(np.isneginf(lse[0, 0, 64:128]))
    rows = [(0, 0, 0), (0, 0, 2), (0, 0, 3)]
    for (b, h, gg), (o, l) in zip(rows, oracle.attn_fwd_groups(to64(Qb), to64(Kb), to64(Vb), fp_, fc_, block, 0.2,
                                                               rows=rows)):
        assert rel_l2(O[0, 0, gg * 64:(gg + 1) * 64], o) <= O_REL_L2
        assert np.max(np.abs(lse[0, 0, gg * 64:(gg + 1) * 64] - l)) <= LSE_MAX_ABS


def test_pipeline_deterministic(dsv):
    w = SMALL["stress_small"]
    x = wl.make_inputs(w, device="cuda")
    outs = []
    for _ in range(2):
        S = dsv.predict_scores(x.Q, x.K, x.Wq, x.Wk, w.block)
        fp, fc, bp, bc = dsv.topk_blocks(S, x.k_per_head, w.block, w.N, w.d)
        O, lse = dsv.sparse_attn_fwd(x.Q, x.K, x.V, fp, fc, w.block)
        outs.append([t.clone() for t in (S, fp, fc, bp, bc, O, lse)])
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_topk_ties_and_special_values(dsv):
    B, H, G, block = 1, 2, 70, 64
    S = torch.randn(B, H, G, G, device="cuda")
    S[0, 0, 0] = 1.0                                   # all tied
    S[0, 0, 1] = 0.0
    S[0, 0, 1, ::2] = -0.0                             # +-0 ties
    S[0, 0, 2, 5] = float("nan")
    S[0, 0, 3, :] = float("-inf")
    S[0, 0, 3, 60] = float("nan")
    S[0, 1, 4] = torch.round(S[0, 1, 4])               # integer-valued, many ties
    ks = [7, 33]
    fp, fc, bp, bc = dsv.topk_blocks(S, ks, block, G * block, 64)
    torch.cuda.synchronize()
    rfp, rfc, rbp, rbc = oracle_lists(to64(S), ks, G)
    assert np.array_equal(fc.cpu().numpy(), rfc) and np.array_equal(fp.cpu().numpy(), rfp)
    assert np.array_equal(bc.cpu().numpy(), rbc) and np.array_equal(bp.cpu().numpy(), rbp)


def test_topk_k_equals_nb_and_one_block(dsv):
    for G, ks in ((33, [33]), (1, [1])):
        S = torch.randn(1, 1, G, G, device="cuda")
        fp, fc, bp, bc = dsv.topk_blocks(S, ks, 128, G * 128, 128)
        torch.cuda.synchronize()
        rfp, rfc, rbp, rbc = oracle_lists(to64(S), ks, G)
        assert np.array_equal(fc.cpu().numpy(), rfc) and np.array_equal(bc.cpu().numpy(), rbc)


def test_empty_problem(dsv):
    z = torch.empty(1, 2, 0, 128, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(2, 128, 16, device="cuda")
    S = dsv.predict_scores(z, z, W, W, 128)
    assert S.shape == (1, 2, 0, 0)
    fp, fc, bp, bc = dsv.topk_blocks(S, [1, 1], 128, 0, 128)
    torch.cuda.synchronize()
    assert fp.cpu().tolist() == [0] and bp.cpu().tolist() == [0]

