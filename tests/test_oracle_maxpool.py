"""Pins of the oracle's max-pooled block scores (CPU only).

The DSV pages ("Technische samenvatting" 2A/2B and the Hindi summary 2A/2B)
score key blocks for a group's proxy query but do not say how a block of keys
is reduced; predict_scores_max is the max-over-the-tile alternative to the
mean reading.  Each test ties it to a fact other than its own form: a tile
worked by hand, the corner closed form of a rank-1 product, the pinned mean
oracle (max >= mean, equal on constant tiles, equal at block 1), and the
symmetries of a bilinear form.  Planted slips at the end must fail them.
"""
import numpy as np

import oracle


def _qk_w(rng, B, H, N, d, r):
    Q, K = rng.standard_normal((2, B, H, N, d))
    Wq, Wk = rng.standard_normal((2, H, d, r))
    return Q, K, Wq, Wk


HAND_Q = np.array([[1, 2], [3, 4], [5, 6], [7, 8]], float)[None, None]
HAND_K = np.array([[1, 0], [0, 1], [2, 2], [0, 0]], float)[None, None]
# token dots q_i . k_l, rows i = 0..3, columns l = 0..3:
#   (1,2): 1 2 6 0 | (3,4): 3 4 14 0 | (5,6): 5 6 22 0 | (7,8): 7 8 30 0
# tile (g, j) of 2 x 2: (0,0) {1,2,3,4} (0,1) {6,0,14,0} (1,0) {5,6,7,8} (1,1) {22,0,30,0}
HAND_MAX = np.array([[4.0, 14.0], [8.0, 30.0]])


def test_maxpool_hand_computed():
    W = np.eye(2)[None]
    S = oracle.predict_scores_max(HAND_Q, HAND_K, W, W, block=2)
    assert np.array_equal(S[0, 0], HAND_MAX)


def test_maxpool_rank_one_corner_closed_form(rng):
    """r = 1: the logit a_i b_l is bilinear, so its maximum over a tile sits
    at a corner of [min a, max a] x [min b, max b]."""
    B, H, N, d, blk = 1, 2, 48, 6, 8
    Q, K, Wq, Wk = _qk_w(rng, B, H, N, d, 1)
    S = oracle.predict_scores_max(Q, K, Wq, Wk, blk)
    G = N // blk
    for h in range(H):
        a = (Q[0, h] @ Wq[h])[:, 0].reshape(G, blk)
        bb = (K[0, h] @ Wk[h])[:, 0].reshape(G, blk)
        for g in range(G):
            for j in range(G):
                corners = [x * y for x in (a[g].min(), a[g].max()) for y in (bb[j].min(), bb[j].max())]
                assert abs(S[0, h, g, j] - max(corners)) <= 1e-12 * (1 + abs(max(corners)))


def test_maxpool_bounds_and_equals_mean_on_constant_tiles(rng):
    B, H, N, d, r, blk = 2, 2, 32, 8, 4, 8
    Q, K, Wq, Wk = _qk_w(rng, B, H, N, d, r)
    Smax = oracle.predict_scores_max(Q, K, Wq, Wk, blk)
    Smean = oracle.predict_scores(Q, K, Wq, Wk, blk)
    assert np.all(Smax >= Smean - 1e-12)
    assert np.any(Smax > Smean + 1e-6)
    # every token of a group (and of a key block) equal: each tile is constant
    Qc = np.repeat(Q[:, :, ::blk], blk, axis=2)
    Kc = np.repeat(K[:, :, ::blk], blk, axis=2)
    np.testing.assert_allclose(oracle.predict_scores_max(Qc, Kc, Wq, Wk, blk),
                               oracle.predict_scores(Qc, Kc, Wq, Wk, blk), rtol=1e-12, atol=1e-12)


def test_maxpool_block_one_is_the_token_logit(rng):
    Q, K, Wq, Wk = _qk_w(rng, 1, 2, 12, 6, 3)
    np.testing.assert_allclose(oracle.predict_scores_max(Q, K, Wq, Wk, 1),
                               oracle.predict_scores(Q, K, Wq, Wk, 1), rtol=1e-12, atol=1e-12)


def test_maxpool_symmetries(rng):
    B, H, N, d, r, blk = 1, 3, 40, 8, 4, 8
    Q, K, Wq, Wk = _qk_w(rng, B, H, N, d, r)
    S = oracle.predict_scores_max(Q, K, Wq, Wk, blk)
    # exchanging the roles of queries and keys transposes every head's score matrix
    St = oracle.predict_scores_max(K, Q, Wk, Wq, blk)
    np.testing.assert_allclose(St, np.swapaxes(S, 2, 3), rtol=1e-12, atol=1e-12)
    # reordering tokens inside every group and block changes nothing
    pq, pk = (np.concatenate([g * blk + rng.permutation(blk) for g in range(N // blk)]) for _ in range(2))
    np.testing.assert_allclose(oracle.predict_scores_max(Q[:, :, pq], K[:, :, pk], Wq, Wk, blk),
                               S, rtol=1e-12, atol=1e-12)
    # a positive factor on one head's W^Q scales that head's scores alone
    Wq2 = Wq.copy()
    Wq2[1] *= 2.5
    S2 = oracle.predict_scores_max(Q, K, Wq2, Wk, blk)
    np.testing.assert_allclose(S2[:, 1], 2.5 * S[:, 1], rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(S2[:, [0, 2]], S[:, [0, 2]])
    # a negative factor turns the maximum into minus the minimum of the tile
    Wq3 = -Wq
    S3 = oracle.predict_scores_max(Q, K, Wq3, Wk, blk)
    L = (Q[0, 0] @ Wq[0]) @ (K[0, 0] @ Wk[0]).T
    G = N // blk
    mins = np.array([[L[g * blk:(g + 1) * blk, j * blk:(j + 1) * blk].min() for j in range(G)] for g in range(G)])
    np.testing.assert_allclose(S3[0, 0], -mins, rtol=1e-12, atol=1e-12)


def test_maxpool_rows_match_full(rng):
    Q, K, Wq, Wk = _qk_w(rng, 2, 2, 32, 8, 4)
    S = oracle.predict_scores_max(Q, K, Wq, Wk, 8)
    rows = [(0, 0, 0), (1, 1, 3), (0, 1, 2), (1, 0, 1)]
    got = oracle.predict_scores_max_rows(Q, K, Wq, Wk, 8, rows)
    for n, (b, h, g) in enumerate(rows):
        np.testing.assert_allclose(got[n], S[b, h, g], rtol=1e-12, atol=1e-12)


def test_maxpool_feeds_both_selections(rng):
    """The selection rules take any score matrix: top-k and mass-threshold
    lists on max-pooled scores obey their invariants."""
    Q, K, Wq, Wk = _qk_w(rng, 1, 2, 64, 8, 4)
    S = oracle.predict_scores_max(Q, K, Wq, Wk, 8)
    ptr, col = oracle.topk_lists(S, [3, 5])
    assert ptr[-1] == 8 * 3 + 8 * 5
    for row in range(16):
        sel = col[ptr[row]:ptr[row + 1]]
        s = S.reshape(16, 8)[row]
        rest = np.setdiff1d(np.arange(8), sel)
        assert np.all(np.diff(sel) > 0) and s[sel].min() >= s[rest].max()
    mptr, mcol = oracle.mass_lists(S, 0.9, 1.0, 1, 8)
    assert np.all(np.diff(mptr) >= 1)


# ------------------------------------------------------------ planted slips

def test_mutants_are_caught():
    W = np.eye(2)[None]

    def mean_not_max(Q, K, Wq, Wk, block):      # the mean reading instead of the max
        return oracle.predict_scores(Q, K, Wq, Wk, block)

    def tiles_misread(Q, K, Wq, Wk, block):     # [N, N] split as [G, G, block, block]
        Q, K = Q[0, 0] @ Wq[0], K[0, 0] @ Wk[0]
        G = Q.shape[0] // block
        return (Q @ K.T).reshape(G, G, block, block).max(axis=(2, 3))[None, None]

    def keys_projected_with_wq(Q, K, Wq, Wk, block):
        return oracle.predict_scores_max(Q, K, Wq, Wq, block)

    for mutant in (mean_not_max, tiles_misread):
        assert not np.array_equal(mutant(HAND_Q, HAND_K, W, W, 2)[0, 0], HAND_MAX)
    rng = np.random.default_rng(9)
    Q, K, Wq, Wk = _qk_w(rng, 1, 1, 16, 4, 1)
    bad = keys_projected_with_wq(Q, K, Wq, Wk, 4)
    a = (Q[0, 0] @ Wq[0])[:, 0].reshape(4, 4)
    b = (K[0, 0] @ Wk[0])[:, 0].reshape(4, 4)
    corner = np.array([[max(x * y for x in (a[g].min(), a[g].max()) for y in (b[j].min(), b[j].max()))
                        for j in range(4)] for g in range(4)])
    assert not np.allclose(bad[0, 0], corner)
