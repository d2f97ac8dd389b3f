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


def _golden_perm(name):
    from pathlib import Path
    lines = [l for l in (Path(__file__).resolve().parent / "golden" / name).read_text().splitlines()
             if l.strip() and not l.startswith("#")]
    return np.array([int(v) for v in lines[0].split()])


def test_mutant_cube_order_slips_are_caught():
    """Plausible slips in the cube token order: the loops inside a cube
    swapped (x before y), the cube extents swapped, the frame stride of the
    raster index wrong; each fails a hand-worked order or the tiling check."""
    def walk(T, Hl, Wl, ct, cy, cx, inner, stride_t):
        perm = []
        for bt in range(T // ct):
            for by in range(Hl // cy):
                for bx in range(Wl // cx):
                    for lt in range(ct):
                        for a in range(cx if inner == "xy" else cy):
                            for b in range(cy if inner == "xy" else cx):
                                ly, lx = (b, a) if inner == "xy" else (a, b)
                                t, y, x = bt * ct + lt, by * cy + ly, bx * cx + lx
                                perm.append(t * stride_t + y * Wl + x)
        return np.array(perm)
    g1 = _golden_perm("cube_order_1x4x4_cube_1x2x2.txt")
    g2 = _golden_perm("cube_order_2x2x4_cube_2x1x2.txt")
    assert np.array_equal(walk(1, 4, 4, 1, 2, 2, "yx", 16), g1)          # the faithful walk passes
    assert not np.array_equal(walk(1, 4, 4, 1, 2, 2, "xy", 16), g1)      # x and y swapped inside a cube
    assert not np.array_equal(walk(2, 2, 4, 2, 1, 2, "yx", 4), g2)       # frame stride Wl instead of Hl*Wl
    swapped = walk(2, 2, 4, 2, 2, 1, "yx", 8)                             # cy and cx swapped
    assert not np.array_equal(swapped, oracle.cube_order(2, 2, 4, 2, 1, 2))


def test_mutant_mass_count_slips_are_caught():
    """Slips in the mass-threshold count: the mass taken without the
    temperature, the count one too small (strict >), and the order by
    ascending score; each disagrees with brute force or a closed form."""
    s = np.full(8, 1.7)
    assert oracle.mass_count_row(s, 0.75, 0.8, 1, 8) == 6                # ceil(0.75 * 8) for equal scores

    def mutant_strict(row, tau, temp):                                   # first count with mass > tau
        p = np.exp(temp * (row - row.max()))
        p /= p.sum()
        cum = np.cumsum(np.sort(p)[::-1])
        return int(np.searchsorted(cum, tau, side="right")) + 1
    assert mutant_strict(s, 0.75, 0.8) != 6

    row = np.array([0.3, 2.0, -1.0, 1.5, 0.9])

    def mutant_no_temp(row, tau):
        p = np.exp(row - row.max())
        p /= p.sum()
        return int(np.searchsorted(np.cumsum(np.sort(p)[::-1]), tau)) + 1
    assert mutant_no_temp(row, 0.9) != oracle.mass_count_row(row, 0.9, 1e3, 1, 5)   # sharp softmax: m = 1

    def mutant_ascending(row, tau, temp):
        p = np.exp(temp * (row - row.max()))
        p /= p.sum()
        return int(np.searchsorted(np.cumsum(np.sort(p)), tau)) + 1
    assert mutant_ascending(row, 0.5, 2.0) != oracle.mass_count_row(row, 0.5, 2.0, 1, 5)
