"""Planted mistakes in copies of oracle routines must fail the pins (CPU only).

Each mutant is a plausible slip (swapped weight, reversed tie rule, dropped
term, transposed operand).  The check that catches it is the same
independent fact used in test_oracle_pins.py.
"""
import math

import numpy as np
import torch

import oracle
from oracle import dsv_oracle as O


def _qkv(rng, B, H, N, d):
    return [rng.standard_normal((B, H, N, d)) for _ in range(3)]


def test_mutant_predictor_wrong_weight_is_caught():
    rng = np.random.default_rng(1)
    Q, K, _ = _qkv(rng, 1, 2, 32, 8)
    Wq, Wk = rng.standard_normal((2, 2, 8, 4))

    def mutant(Q, K, Wq, Wk, block):            # projects keys with W^Q
        return oracle.predict_scores(Q, K, Wq, Wq, block)
    S = mutant(Q, K, Wq, Wk, 8)
    L = (Q[0, 0] @ Wq[0]) @ (K[0, 0] @ Wk[0]).T
    brute = L.reshape(4, 8, 4, 8).mean(axis=(1, 3))
    assert not np.allclose(S[0, 0], brute)


def test_mutant_tie_toward_higher_index_is_caught():
    row = np.array([1.0, 3.0, 3.0, 0.0, 3.0])

    def mutant(s, k):                           # ties resolved toward the higher index
        order = sorted(range(len(s)), key=lambda j: (-s[j], -j))
        return sorted(order[:k])
    assert mutant(row, 2) != [1, 2]
    assert oracle.topk_row(row, 2).tolist() == [1, 2]


def test_mutant_missing_scale_is_caught():
    rng = np.random.default_rng(2)
    Q, K, V = _qkv(rng, 1, 1, 32, 16)
    mask = np.ones((1, 1, 2, 2), bool)
    bad, _ = oracle.attn_fwd_masked(Q, K, V, mask, 16, scale=1.0)   # scale 1 instead of 1/sqrt(d)
    ref = torch.nn.functional.scaled_dot_product_attention(*(torch.from_numpy(x) for x in (Q, K, V))).numpy()
    assert np.max(np.abs(bad - ref)) > 1e-3


def _autograd(Q, K, V, dO, mask, blk):
    tm = np.repeat(np.repeat(mask, blk, axis=2), blk, axis=3)
    q, k, v = (torch.tensor(x, requires_grad=True) for x in (Q, K, V))
    torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=torch.from_numpy(tm)).backward(torch.from_numpy(dO))
    return q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


def test_mutant_backward_slips_are_caught(monkeypatch):
    rng = np.random.default_rng(3)
    B, H, N, d, blk = 1, 1, 32, 8, 8
    Q, K, V = _qkv(rng, B, H, N, d)
    dO = rng.standard_normal((B, H, N, d))
    ptr = np.arange(0, 4 * 2 + 1, 2)
    col = np.array([0, 2, 1, 3, 0, 1, 2, 3])
    mask = oracle.block_mask(ptr, col, B, H, 4, 4)
    ref = _autograd(Q, K, V, dO, mask, blk)

    def no_D(q, kk, vv, do, tau):               # drops the D_i term of dS
        s = tau * (q @ kk.T)
        P = np.exp(s - s.max(1, keepdims=True))
        P /= P.sum(1, keepdims=True)
        dS = P * (do @ vv.T)
        return tau * (dS @ kk), tau * (dS.T @ q), P.T @ do

    def dp_from_keys(q, kk, vv, do, tau):      # dP = dO K^T instead of dO V^T
        s = tau * (q @ kk.T)
        P = np.exp(s - s.max(1, keepdims=True))
        P /= P.sum(1, keepdims=True)
        dP = do @ kk.T
        dS = P * (dP - (P * dP).sum(1, keepdims=True))
        return tau * (dS @ kk), tau * (dS.T @ q), P.T @ do

    _orig = O._group_bwd
    for mutant, which in ((no_D, 0), (dp_from_keys, 1)):
        monkeypatch.setattr(O, "_group_bwd", mutant)
        got = oracle.attn_bwd_groups(Q, K, V, dO, ptr, col, blk)
        assert np.max(np.abs(got[which] - ref[which])) > 1e-6
        monkeypatch.setattr(O, "_group_bwd", _orig)
    got = oracle.attn_bwd_groups(Q, K, V, dO, ptr, col, blk)
    for a, r in zip(got, ref):
        assert np.max(np.abs(a - r)) <= 1e-11
