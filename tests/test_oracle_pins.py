"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test ties one oracle function to an independent fact: a hand-computed
closed form, brute force over all subsets, a library routine (torch fp64
scaled_dot_product_attention and autograd), central finite differences, or an
invariant the mathematics fixes.  The pages print no worked example, so no
stored golden values exist (see tests/golden/README.md).
"""
import itertools
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from conftest import rel_l2


def _rand_qkv(rng, B, H, N, d, scale=1.0):
    return [rng.standard_normal((B, H, N, d)) * scale for _ in range(3)]


def _random_lists(rng, B, H, G, nb, ks):
    ptr = [0]
    col = []
    for b in range(B):
        for h in range(H):
            for g in range(G):
                sel = np.sort(rng.choice(nb, size=ks[h], replace=False))
                col.extend(sel.tolist())
                ptr.append(ptr[-1] + ks[h])
    return np.array(ptr), np.array(col)


# ------------------------------------------------------------------ predictor

def test_predictor_hand_computed():
    """beta=2, d=r=2, W=I: S = mean(Q_g) . mean(K_j), worked by hand."""
    Q = np.array([[1, 2], [3, 4], [5, 6], [7, 8]], float)[None, None]
    K = np.array([[1, 0], [0, 1], [2, 2], [0, 0]], float)[None, None]
    W = np.eye(2)[None]
    # qbar_0 = (2,3), qbar_1 = (6,7); kbar_0 = (.5,.5), kbar_1 = (1,1)
    expect = np.array([[2.5, 5.0], [6.5, 13.0]])
    S = oracle.predict_scores(Q, K, W, W, block=2)
    assert np.array_equal(S[0, 0], expect)


def test_predictor_equals_mean_of_lowrank_logit_tile(rng):
    """S[g, j] is the mean of the block x block tile of (Q Wq)(K Wk)^T."""
    B, H, N, d, r, blk = 2, 3, 32, 8, 4, 8
    Q, K, _ = _rand_qkv(rng, B, H, N, d)
    Wq = rng.standard_normal((H, d, r))
    Wk = rng.standard_normal((H, d, r))
    S = oracle.predict_scores(Q, K, Wq, Wk, blk)
    G = N // blk
    for b in range(B):
        for h in range(H):
            L = (Q[b, h] @ Wq[h]) @ (K[b, h] @ Wk[h]).T
            brute = np.array([[L[g * blk:(g + 1) * blk, j * blk:(j + 1) * blk].mean()
                               for j in range(G)] for g in range(G)])
            assert np.allclose(S[b, h], brute, rtol=1e-12, atol=1e-12)


def test_predictor_pool_first_equals_project_first(rng):
    Q, K, _ = _rand_qkv(rng, 1, 2, 64, 16)
    Wq = rng.standard_normal((2, 16, 8))
    Wk = rng.standard_normal((2, 16, 8))
    a = oracle.predict_scores(Q, K, Wq, Wk, 16)
    b = oracle.predict_scores_pool_first(Q, K, Wq, Wk, 16)
    assert np.max(np.abs(a - b)) <= 1e-12 * np.max(np.abs(a))


def test_predictor_uses_each_heads_own_weights(rng):
    """Zero predictor weights on head 1 only => head 1 scores are exactly 0."""
    Q, K, _ = _rand_qkv(rng, 1, 2, 32, 8)
    Wq = rng.standard_normal((2, 8, 4))
    Wk = rng.standard_normal((2, 8, 4))
    Wk[1] = 0.0
    S = oracle.predict_scores(Q, K, Wq, Wk, 8)
    assert np.all(S[0, 1] == 0.0) and np.all(S[0, 0] != 0.0)


def test_predictor_rows_match_full(rng):
    Q, K, _ = _rand_qkv(rng, 2, 2, 48, 8)
    Wq = rng.standard_normal((2, 8, 4))
    Wk = rng.standard_normal((2, 8, 4))
    S = oracle.predict_scores(Q, K, Wq, Wk, 8)
    rows = [(0, 1, 3), (1, 0, 0), (1, 1, 5)]
    R = oracle.predict_scores_rows(Q, K, Wq, Wk, 8, rows)
    for n, (b, h, g) in enumerate(rows):
        assert np.allclose(R[n], S[b, h, g], rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------------- top-k

def _brute_topk(row, k):
    """Max-sum k-subset, ties toward the lexicographically smallest index list."""
    vals = [Fraction(v) for v in row]
    best = None
    for sub in itertools.combinations(range(len(row)), k):   # lexicographic order
        s = sum(vals[i] for i in sub)
        if best is None or s > best[0]:
            best = (s, sub)
    return list(best[1])


def test_topk_brute_force_with_ties(rng):
    for nb in range(1, 8):
        for _ in range(20):
            row = rng.integers(-3, 4, size=nb).astype(float)   # many exact ties
            for k in range(1, nb + 1):
                assert oracle.topk_row(row, k).tolist() == _brute_topk(row, k)


def test_topk_brute_force_random(rng):
    for _ in range(50):
        row = rng.standard_normal(7)
        for k in range(1, 8):
            assert oracle.topk_row(row, k).tolist() == _brute_topk(row, k)


def test_topk_constructed_ties():
    assert oracle.topk_row([0.0, -0.0, 0.0, -0.0], 2).tolist() == [0, 1]
    assert oracle.topk_row([-0.0, 0.0, 1.0], 2).tolist() == [0, 2]
    assert oracle.topk_row([5.0, 1.0, 5.0, 5.0], 2).tolist() == [0, 2]
    assert oracle.topk_row([2.0] * 9, 4).tolist() == [0, 1, 2, 3]
    assert oracle.topk_row([np.nan, 1.0, 2.0, np.nan], 3).tolist() == [0, 1, 2]
    assert oracle.topk_row([-np.inf, np.nan, -1.0], 2).tolist() == [0, 2]
    assert oracle.topk_row([np.nan, -np.inf], 1).tolist() == [1]          # NaN below -inf
    assert oracle.topk_row([np.nan, -np.inf, np.nan, -np.inf], 3).tolist() == [0, 1, 3]


def test_topk_lists_invariants(rng):
    B, H, G = 2, 3, 37
    S = rng.standard_normal((B, H, G, G)).astype(np.float32).astype(np.float64)
    S[0, 0, 0, :] = 1.0                                     # an all-tied row
    ks = [1, 5, 37]
    ptr, col = oracle.topk_lists(S, ks)
    assert ptr[-1] == B * G * sum(ks) == len(col)
    for b in range(B):
        for h in range(H):
            for g in range(G):
                row = (b * H + h) * G + g
                sel = col[ptr[row]:ptr[row + 1]]
                assert len(sel) == ks[h] and np.all(np.diff(sel) > 0)
                uns = np.setdiff1d(np.arange(G), sel)
                if len(uns):
                    assert S[b, h, g, sel].min() >= S[b, h, g, uns].max()
                    # an unselected index equal to the threshold lies above every selected one of that value
                    t = S[b, h, g, sel].min()
                    eq_uns = uns[S[b, h, g, uns] == t]
                    eq_sel = sel[S[b, h, g, sel] == t]
                    if len(eq_uns):
                        assert eq_uns.min() > eq_sel.max()
                assert sel.tolist() == oracle.topk_row(S[b, h, g], ks[h]).tolist()
    assert col[:1].tolist() == [0]


def test_transpose_is_exact_transpose(rng):
    B, H, G = 2, 2, 23
    ks = [4, 9]
    ptr, col = _random_lists(rng, B, H, G, G, ks)
    bptr, bcol = oracle.transpose_lists(ptr, col, B, H, G, G)
    m = oracle.block_mask(ptr, col, B, H, G, G)
    assert bptr[-1] == ptr[-1]
    for b in range(B):
        for h in range(H):
            for j in range(G):
                r = (b * H + h) * G + j
                assert bcol[bptr[r]:bptr[r + 1]].tolist() == np.nonzero(m[b, h, :, j])[0].tolist()


# ---------------------------------------------------------- attention forward

def _sdpa(Q, K, V, tok_mask, scale):
    q, k, v = (torch.from_numpy(np.ascontiguousarray(x)) for x in (Q, K, V))
    m = None if tok_mask is None else torch.from_numpy(tok_mask)
    return torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=m, scale=scale).numpy()


def _tok_mask(mask, blk):
    return np.repeat(np.repeat(mask, blk, axis=2), blk, axis=3)


def test_fwd_all_blocks_equals_dense_sdpa(rng):
    B, H, N, d, blk = 1, 2, 64, 16, 16
    Q, K, V = _rand_qkv(rng, B, H, N, d)
    G = N // blk
    mask = np.ones((B, H, G, G), bool)
    O, L = oracle.attn_fwd_masked(Q, K, V, mask, blk)
    ref = _sdpa(Q, K, V, None, 1 / math.sqrt(d))
    assert np.max(np.abs(O - ref)) <= 1e-12
    s = (Q @ np.swapaxes(K, 2, 3)) / math.sqrt(d)
    lse = np.log(np.exp(s).sum(-1))
    assert np.max(np.abs(L - lse)) <= 1e-12


def test_fwd_masked_equals_sdpa_with_block_mask(rng):
    B, H, N, d, blk = 2, 2, 96, 8, 16
    G = N // blk
    Q, K, V = _rand_qkv(rng, B, H, N, d, scale=2.0)
    ptr, col = _random_lists(rng, B, H, G, G, [2, 4])
    mask = oracle.block_mask(ptr, col, B, H, G, G)
    O, L = oracle.attn_fwd_masked(Q, K, V, mask, blk, scale=0.3)
    ref = _sdpa(Q, K, V, _tok_mask(mask, blk), 0.3)
    assert np.max(np.abs(O - ref)) <= 1e-12 * max(1.0, np.abs(ref).max())
    Og, Lg = oracle.attn_fwd_groups(Q, K, V, ptr, col, blk, scale=0.3)
    assert np.max(np.abs(Og - O)) <= 1e-12 and np.max(np.abs(Lg - L)) <= 1e-12
    rows = [(1, 0, 2), (0, 1, 5)]
    for (b, h, g), (o, l) in zip(rows, oracle.attn_fwd_groups(Q, K, V, ptr, col, blk, 0.3, rows=rows)):
        assert np.array_equal(o, Og[b, h, g * blk:(g + 1) * blk])


def test_fwd_rows_of_p_sum_to_one_and_lse_bounds(rng):
    B, H, N, d, blk = 1, 2, 64, 8, 8
    G = N // blk
    Q, K, V = _rand_qkv(rng, B, H, N, d, scale=3.0)
    ptr, col = _random_lists(rng, B, H, G, G, [3, 1])
    mask = oracle.block_mask(ptr, col, B, H, G, G)
    _, L = oracle.attn_fwd_masked(Q, K, V, mask, blk)
    tm = _tok_mask(mask, blk)
    s = (Q @ np.swapaxes(K, 2, 3)) / math.sqrt(d)
    P = np.where(tm, np.exp(s - L[..., None]), 0.0)
    assert np.max(np.abs(P.sum(-1) - 1.0)) <= 1e-12
    smax = np.where(tm, s, -np.inf).max(-1)
    nkeys = tm.sum(-1)
    assert np.all(L >= smax) and np.all(L <= smax + np.log(nkeys) + 1e-12)


def test_fwd_constant_values_and_key_shift_invariance(rng):
    B, H, N, d, blk = 1, 1, 48, 8, 8
    G = N // blk
    Q, K, V = _rand_qkv(rng, B, H, N, d)
    ptr, col = _random_lists(rng, B, H, G, G, [2])
    mask = oracle.block_mask(ptr, col, B, H, G, G)
    c = rng.standard_normal(d)
    O, _ = oracle.attn_fwd_masked(Q, K, np.broadcast_to(c, V.shape), mask, blk)
    assert np.max(np.abs(O - c)) <= 1e-12
    O0, L0 = oracle.attn_fwd_masked(Q, K, V, mask, blk)
    u = rng.standard_normal(d)
    O1, L1 = oracle.attn_fwd_masked(Q, K + u, V, mask, blk)
    assert np.max(np.abs(O1 - O0)) <= 1e-11
    assert np.max(np.abs(L1 - L0 - (Q @ u) / math.sqrt(d))) <= 1e-11


# --------------------------------------------------------- attention backward

def test_bwd_finite_differences():
    rng = np.random.default_rng(7)
    B, H, N, d, blk = 1, 2, 16, 4, 4
    G = N // blk
    Q, K, V = _rand_qkv(rng, B, H, N, d)
    dO = rng.standard_normal((B, H, N, d))
    ptr, col = _random_lists(rng, B, H, G, G, [2, 3])
    mask = oracle.block_mask(ptr, col, B, H, G, G)
    dQ, dK, dV = oracle.attn_bwd_masked(Q, K, V, dO, mask, blk)
    eps = 1e-6

    def loss(q, k, v):
        return float((oracle.attn_fwd_masked(q, k, v, mask, blk)[0] * dO).sum())

    for which, grad in ((0, dQ), (1, dK), (2, dV)):
        num = np.zeros_like(grad)
        for idx in np.ndindex(*grad.shape):
            args = [Q.copy(), K.copy(), V.copy()]
            args[which][idx] += eps
            up = loss(*args)
            args[which][idx] -= 2 * eps
            dn = loss(*args)
            num[idx] = (up - dn) / (2 * eps)
        assert np.max(np.abs(num - grad)) <= 1e-6 * max(1.0, np.abs(grad).max())


def test_bwd_equals_torch_autograd(rng):
    B, H, N, d, blk = 1, 2, 128, 16, 16
    G = N // blk
    Q, K, V = _rand_qkv(rng, B, H, N, d, scale=1.5)
    dO = rng.standard_normal((B, H, N, d))
    ptr, col = _random_lists(rng, B, H, G, G, [3, 5])
    mask = oracle.block_mask(ptr, col, B, H, G, G)
    dQ, dK, dV = oracle.attn_bwd_masked(Q, K, V, dO, mask, blk)
    q, k, v = (torch.tensor(x, requires_grad=True) for x in (Q, K, V))
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=torch.from_numpy(_tok_mask(mask, blk)))
    o.backward(torch.from_numpy(dO))
    for ours, ref in ((dQ, q.grad), (dK, k.grad), (dV, v.grad)):
        assert np.max(np.abs(ours - ref.numpy())) <= 1e-11 * max(1.0, ref.abs().max().item())


def test_bwd_invariants_and_group_forms(rng):
    B, H, N, d, blk = 2, 2, 80, 8, 8
    G = N // blk
    Q, K, V = _rand_qkv(rng, B, H, N, d, scale=2.0)
    dO = rng.standard_normal((B, H, N, d))
    ptr, col = _random_lists(rng, B, H, G, G, [2, 4])
    mask = oracle.block_mask(ptr, col, B, H, G, G)
    dQ, dK, dV = oracle.attn_bwd_masked(Q, K, V, dO, mask, blk)
    # a shift shared by every key moves each row's logits uniformly
    assert np.max(np.abs(dK.sum(axis=2))) <= 1e-11
    # every row of P sums to one
    assert np.max(np.abs(dV.sum(axis=2) - dO.sum(axis=2))) <= 1e-11
    unsel = ~mask.any(axis=2)                                  # [B,H,nb] blocks nobody chose
    for b, h, j in zip(*np.nonzero(unsel)):
        assert np.all(dK[b, h, j * blk:(j + 1) * blk] == 0) and np.all(dV[b, h, j * blk:(j + 1) * blk] == 0)
    gQ, gK, gV = oracle.attn_bwd_groups(Q, K, V, dO, ptr, col, blk)
    for a, c in ((gQ, dQ), (gK, dK), (gV, dV)):
        assert np.max(np.abs(a - c)) <= 1e-12 * max(1.0, np.abs(c).max())
    bptr, bcol = oracle.transpose_lists(ptr, col, B, H, G, G)
    blocks = [(0, 0, 1), (1, 1, 7), (1, 0, 9)]
    for (b, h, j), (dk, dv) in zip(blocks, oracle.attn_bwd_kv_blocks(Q, K, V, dO, ptr, col, bptr, bcol, blk, blocks)):
        assert np.allclose(dk, dK[b, h, j * blk:(j + 1) * blk], atol=1e-12)
        assert np.allclose(dv, dV[b, h, j * blk:(j + 1) * blk], atol=1e-12)
    rows = [(0, 1, 3), (1, 0, 0)]
    for (b, h, g), dq in zip(rows, oracle.attn_bwd_dq_rows(Q, K, V, dO, ptr, col, blk, rows)):
        assert np.allclose(dq, dQ[b, h, g * blk:(g + 1) * blk], atol=1e-12)


def test_bwd_kv_blocks_given_stats_equals_closed_form(rng):
    """The block form fed each row's LSE and D gives the closed-form dK/dV
    of attn_bwd_masked (itself pinned to torch autograd and finite
    differences); LSE and D are taken from their definitions over the
    masked rows, not from the GPU."""
    B, H, N, d, blk = 2, 2, 96, 8, 8
    G = N // blk
    Q, K, V = _rand_qkv(rng, B, H, N, d, scale=2.0)
    dO = rng.standard_normal((B, H, N, d))
    ptr, col = _random_lists(rng, B, H, G, G, [3, 7])
    mask = oracle.block_mask(ptr, col, B, H, G, G)
    O, lse = oracle.attn_fwd_masked(Q, K, V, mask, blk)
    _, dK, dV = oracle.attn_bwd_masked(Q, K, V, dO, mask, blk)
    # D_i = sum_j P_ij dP_ij over the masked row, written out from P and dP
    tau = 1.0 / math.sqrt(d)
    D = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            tok = np.repeat(np.repeat(mask[b, h], blk, axis=0), blk, axis=1)
            P = np.where(tok, np.exp(tau * Q[b, h] @ K[b, h].T - lse[b, h][:, None]), 0.0)
            D[b, h] = (P * (dO[b, h] @ V[b, h].T)).sum(axis=1)
    assert np.allclose(D, (dO * O).sum(axis=3), atol=1e-12)     # the rowsum(dO * O) identity
    bptr, bcol = oracle.transpose_lists(ptr, col, B, H, G, G)
    blocks = [(b, h, j) for b in range(B) for h in range(H) for j in range(G)]
    got = oracle.attn_bwd_kv_blocks_given_stats(Q, K, V, dO, lse, D, bptr, bcol, blk, blocks)
    for (b, h, j), (dk, dv) in zip(blocks, got):
        sl = slice(j * blk, (j + 1) * blk)
        assert np.max(np.abs(dk - dK[b, h, sl])) <= 1e-12 * max(1.0, np.abs(dK).max())
        assert np.max(np.abs(dv - dV[b, h, sl])) <= 1e-12 * max(1.0, np.abs(dV).max())
    # each statistic matters: a shifted LSE or a dropped D moves the result
    bad_l = oracle.attn_bwd_kv_blocks_given_stats(Q, K, V, dO, lse + 0.1, D, bptr, bcol, blk, blocks[:4])
    bad_d = oracle.attn_bwd_kv_blocks_given_stats(Q, K, V, dO, lse, 0 * D, bptr, bcol, blk, blocks[:4])
    for (b, h, j), (dk, dv), (dk2, _) in zip(blocks[:4], bad_l, bad_d):
        sl = slice(j * blk, (j + 1) * blk)
        if np.abs(dV[b, h, sl]).max() > 0:
            assert np.max(np.abs(dv - dV[b, h, sl])) > 1e-3
            assert np.max(np.abs(dk2 - dK[b, h, sl])) > 1e-3
