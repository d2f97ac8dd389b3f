"""fp64 CPU oracle for the DSV dynamic sparse 3D attention hot path.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check of
``__graft_entry__`` and the ``cpu_baseline`` / reference leg of ``bench.py``
may import this module.  The product path (the CUDA library and its Python
binding) never calls it, and it shares no code, tables or helpers with the
CUDA sources.

Source pages (cited by title and section):
  [nl] "DSV: Exploiting Dynamic Sparsity to Accelerate Large-Scale Video DiT
       Training", gist.science/nl/paper/2502.07590, "Technische samenvatting".
  [hi] the same title, gist.science/hi/paper/2502.07590, technical summary.

What the pages fix, and the reading taken where they are silent:
  * Predictor ([nl] 2A, [hi] 2A): per-head low-rank matrices W^Q_lr, W^K_lr
    (rank d_lr << d_k) whose product Q_lr K_lr^T approximates Q K^T.
  * Query grouping ([nl] 2B, [hi] 2B): adjacent tokens share one proxy
    query's critical-KV indices.  Reading: a group is `block` consecutive
    tokens; its proxy is the mean of its low-rank queries; a key block is
    scored by the mean of its low-rank keys; score = plain dot product (no
    scale; a positive scale cannot change a top-k).
  * Selection ([nl] 2B, [hi] 2A/2B): top-k critical KV blocks per group.
    Reading: k per head, ties broken toward the lower block index.
  * Sparse attention ([nl] 2A, [hi] 2A): softmax attention evaluated only over
    the selected KV.  Reading: scale 1/sqrt(d) unless given, natural-log LSE,
    bidirectional (no causal mask), no forced blocks.
  * Backward: the pages train with it ([nl] 2A stage 2); the gradient is the
    ordinary softmax-attention gradient restricted to the same mask.
  * Mass-threshold selection ([nl] 2A, [hi] 2A: the critical KV carry about
    90 % of the attention score).  Reading: block masses are the softmax of
    temperature * S over the row; the smallest top set reaching tau is kept,
    clamped to [kmin, kmax]; a row with a non-finite score keeps kmax.
  * Max-pooled block scores ([nl] 2A, 2B: the pages do not say how a tile of
    low-rank logits becomes one score).  Reading, as the alternative to the
    mean: the largest logit (Q_i W^Q) . (K_l W^K) over the group's query
    tokens i and the block's key tokens l, no scale.
  * 3D cube grouping ([nl] 2B, [hi] 2B: queries grouped in small cubes).
    Reading: a token permutation making every run of `block` tokens one
    ct x cy x cx cube (cube grid and cube interior both in raster order).

Every function works in float64 on numpy arrays.  Shapes:
  Q, K, V, dO : [B, H, N, d];  Wq, Wk : [H, d, r];  S : [B, H, G, nb]
  fwd CSR: ptr [B*H*G + 1], col [nnz] (block index j within its (b, h));
  bwd CSR: ptr [B*H*nb + 1], col [nnz] (group index g within its (b, h)).
"""
from __future__ import annotations

import math
from typing import Iterable, List, Optional, Sequence, Tuple

import numpy as np


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


# --------------------------------------------------------------------------
# Predictor ([nl] 2A low-rank predictor, 2B query grouping)
# --------------------------------------------------------------------------

def predict_scores(Q, K, Wq, Wk, block: int) -> np.ndarray:
    """Block scores S[b,h,g,j] = qbar_g . kbar_j, literal project-then-pool.

    Q_lr = Q W^Q_lr[h] and K_lr = K W^K_lr[h] for every token; qbar_g is the
    mean of Q_lr over the `block` tokens of group g, kbar_j the mean of K_lr
    over key block j.
    """
    Q, K, Wq, Wk = _f64(Q), _f64(K), _f64(Wq), _f64(Wk)
    B, H, N, d = Q.shape
    G = N // block
    r = Wq.shape[2]
    S = np.empty((B, H, G, G), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            q_lr = Q[b, h] @ Wq[h]                  # [N, r]
            k_lr = K[b, h] @ Wk[h]
            qbar = q_lr.reshape(G, block, r).mean(axis=1)
            kbar = k_lr.reshape(G, block, r).mean(axis=1)
            S[b, h] = qbar @ kbar.T
    return S


def predict_scores_rows(Q, K, Wq, Wk, block: int, rows: Sequence[Tuple[int, int, int]]) -> np.ndarray:
    """Rows S[b,h,g,:] for the listed (b, h, g), same definition as predict_scores."""
    Wq, Wk = _f64(Wq), _f64(Wk)
    B, H, N, d = Q.shape
    G = N // block
    r = Wq.shape[2]
    out = np.empty((len(rows), G), dtype=np.float64)
    kbar_cache = {}
    for n, (b, h, g) in enumerate(rows):
        if (b, h) not in kbar_cache:
            k_lr = _f64(K[b, h]) @ Wk[h]
            kbar_cache[(b, h)] = k_lr.reshape(G, block, r).mean(axis=1)
        q_lr = _f64(Q[b, h, g * block:(g + 1) * block]) @ Wq[h]
        out[n] = kbar_cache[(b, h)] @ q_lr.mean(axis=0)
    return out


def predict_scores_pool_first(Q, K, Wq, Wk, block: int) -> np.ndarray:
    """The same scores with pooling before projection (equal by linearity).

    Used only as a pin of predict_scores, never as the oracle.
    """
    Q, K, Wq, Wk = _f64(Q), _f64(K), _f64(Wq), _f64(Wk)
    B, H, N, d = Q.shape
    G = N // block
    S = np.empty((B, H, G, G))
    for b in range(B):
        for h in range(H):
            qm = Q[b, h].reshape(G, block, d).mean(axis=1) @ Wq[h]
            km = K[b, h].reshape(G, block, d).mean(axis=1) @ Wk[h]
            S[b, h] = qm @ km.T
    return S


def predict_scores_max(Q, K, Wq, Wk, block: int) -> np.ndarray:
    """Max-pooled block scores: S[b,h,g,j] = the largest low-rank logit
    Q_lr[i] . K_lr[l] over the query tokens i of group g and the key tokens l
    of block j (no scale).

    The pages do not say how a block is scored; this is the alternative to the
    mean reading (predict_scores), which is the mean of the same tile.  The
    whole [N, N] low-rank logit matrix of one (b, h) is formed, then each
    block x block tile is reduced by its maximum.
    """
    Q, K, Wq, Wk = _f64(Q), _f64(K), _f64(Wq), _f64(Wk)
    B, H, N, d = Q.shape
    G = N // block
    S = np.empty((B, H, G, G), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            L = (Q[b, h] @ Wq[h]) @ (K[b, h] @ Wk[h]).T      # [N, N] low-rank logits
            S[b, h] = L.reshape(G, block, G, block).max(axis=(1, 3))
    return S


def predict_scores_max_rows(Q, K, Wq, Wk, block: int, rows: Sequence[Tuple[int, int, int]]) -> np.ndarray:
    """Rows S[b,h,g,:] of predict_scores_max for the listed (b, h, g)."""
    Wq, Wk = _f64(Wq), _f64(Wk)
    B, H, N, d = Q.shape
    G = N // block
    out = np.empty((len(rows), G), dtype=np.float64)
    k_cache = {}
    for n, (b, h, g) in enumerate(rows):
        if (b, h) not in k_cache:
            k_cache[(b, h)] = _f64(K[b, h]) @ Wk[h]                # [N, r]
        q_lr = _f64(Q[b, h, g * block:(g + 1) * block]) @ Wq[h]   # [block, r]
        L = q_lr @ k_cache[(b, h)].T                              # [block, N]
        out[n] = L.reshape(block, G, block).max(axis=(0, 2))
    return out


# --------------------------------------------------------------------------
# Top-k selection and the transposed lists ([nl] 2B, [hi] 2B)
# --------------------------------------------------------------------------

def topk_row(scores_row, k: int) -> np.ndarray:
    """The k block indices with the largest scores, ascending.

    Total order: larger score first, equal scores by lower index; -0.0 and
    +0.0 compare equal; NaN ranks below every number.
    """
    return np.sort(_rank_order(_f64(scores_row)[None, :])[0, :k])


def _rank_order(S2: np.ndarray) -> np.ndarray:
    """Per row, indices from best to worst under the total order above."""
    nan = np.isnan(S2)
    key = np.where(nan, np.inf, -S2)                           # larger score first
    order = np.argsort(key, axis=1, kind="stable")            # stable => lower index first on ties
    # NaN after every number, -inf included (second stable pass keeps index order)
    back = np.argsort(np.take_along_axis(nan, order, axis=1), axis=1, kind="stable")
    return np.take_along_axis(order, back, axis=1)


def topk_lists(S, k_per_head: Sequence[int]) -> Tuple[np.ndarray, np.ndarray]:
    """Forward CSR over all rows (b, h, g): ptr [B*H*G+1], col [nnz]."""
    S = _f64(S)
    B, H, G, nb = S.shape
    ptr = np.zeros(B * H * G + 1, dtype=np.int64)
    cols: List[np.ndarray] = []
    row = 0
    for b in range(B):
        for h in range(H):
            k = int(k_per_head[h])
            sel = np.sort(_rank_order(S[b, h])[:, :k], axis=1)
            for g in range(G):
                cols.append(sel[g])
                ptr[row + 1] = ptr[row] + k
                row += 1
    col = np.concatenate(cols).astype(np.int64) if cols else np.zeros(0, np.int64)
    return ptr, col


def transpose_lists(fwd_ptr, fwd_col, B: int, H: int, G: int, nb: int) -> Tuple[np.ndarray, np.ndarray]:
    """Backward CSR: for each (b, h, j) the ascending groups g whose list holds j."""
    fwd_ptr = np.asarray(fwd_ptr, dtype=np.int64)
    fwd_col = np.asarray(fwd_col, dtype=np.int64)
    lists: List[List[int]] = [[] for _ in range(B * H * nb)]
    for bh in range(B * H):
        for g in range(G):
            row = bh * G + g
            for j in fwd_col[fwd_ptr[row]:fwd_ptr[row + 1]]:
                lists[bh * nb + int(j)].append(g)      # g visited ascending
    ptr = np.zeros(B * H * nb + 1, dtype=np.int64)
    for i, l in enumerate(lists):
        ptr[i + 1] = ptr[i] + len(l)
    col = np.array([g for l in lists for g in l], dtype=np.int64)
    return ptr, col


def block_mask(fwd_ptr, fwd_col, B: int, H: int, G: int, nb: int) -> np.ndarray:
    """Boolean [B, H, G, nb]: True where block j is in group g's list."""
    m = np.zeros((B, H, G, nb), dtype=bool)
    for b in range(B):
        for h in range(H):
            for g in range(G):
                row = (b * H + h) * G + g
                m[b, h, g, fwd_col[fwd_ptr[row]:fwd_ptr[row + 1]]] = True
    return m


# --------------------------------------------------------------------------
# Sparse attention forward ([nl] 2A stage 2, [hi] 2A critical-KV attention)
# --------------------------------------------------------------------------

def _scale(d: int, scale: Optional[float]) -> float:
    return 1.0 / math.sqrt(d) if not scale else float(scale)


def attn_fwd_masked(Q, K, V, mask, block: int, scale: Optional[float] = None):
    """Literal masked softmax attention: every row over all N keys.

    s_ij = scale * q_i . k_j where block(j) is in group(i)'s list, -inf
    elsewhere; O_i = sum_j softmax(s_i)_j v_j; LSE_i = ln sum_j exp(s_ij).
    Returns O [B,H,N,d] and LSE [B,H,N].
    """
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, H, N, d = Q.shape
    tau = _scale(d, scale)
    O = np.empty_like(Q)
    LSE = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            tok_mask = np.repeat(np.repeat(mask[b, h], block, axis=0), block, axis=1)
            s = tau * (Q[b, h] @ K[b, h].T)
            s = np.where(tok_mask, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            e = np.exp(s - m)
            l = e.sum(axis=1, keepdims=True)
            O[b, h] = (e @ V[b, h]) / l
            LSE[b, h] = (m + np.log(l))[:, 0]
    return O, LSE


def _group_keys(cols, block: int) -> np.ndarray:
    return (np.asarray(cols, dtype=np.int64)[:, None] * block + np.arange(block)[None, :]).reshape(-1)


def attn_fwd_groups(Q, K, V, fwd_ptr, fwd_col, block: int, scale: Optional[float] = None,
                    rows: Optional[Iterable[Tuple[int, int, int]]] = None):
    """Masked attention for whole groups, summing only over the selected keys.

    Same definition as attn_fwd_masked: the keys outside the mask carry
    exp(-inf) = 0, so they are left out of the sums.  With rows=None every
    group is evaluated and full [B,H,N,d] / [B,H,N] arrays are returned;
    otherwise a list of (O_g [block,d], LSE_g [block]) in the order of rows.
    """
    B, H, N, d = Q.shape
    G = N // block
    tau = _scale(d, scale)
    full = rows is None
    if full:
        rows = [(b, h, g) for b in range(B) for h in range(H) for g in range(G)]
        O = np.empty((B, H, N, d))
        LSE = np.empty((B, H, N))
    res = []
    for (b, h, g) in rows:
        row = (b * H + h) * G + g
        keys = _group_keys(fwd_col[fwd_ptr[row]:fwd_ptr[row + 1]], block)
        q = _f64(Q[b, h, g * block:(g + 1) * block])
        s = tau * (q @ _f64(K[b, h, keys]).T)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        l = e.sum(axis=1, keepdims=True)
        o = (e @ _f64(V[b, h, keys])) / l
        lse = (m + np.log(l))[:, 0]
        if full:
            O[b, h, g * block:(g + 1) * block] = o
            LSE[b, h, g * block:(g + 1) * block] = lse
        else:
            res.append((o, lse))
    return (O, LSE) if full else res


# --------------------------------------------------------------------------
# Sparse attention backward (gradient of the masked softmax attention)
# --------------------------------------------------------------------------

def attn_bwd_masked(Q, K, V, dO, mask, block: int, scale: Optional[float] = None):
    """Closed-form gradient of L = sum(dO * O) through attn_fwd_masked.

    P = softmax rows; dV = P^T dO; dP = dO V^T; D_i = sum_j P_ij dP_ij;
    dS = P * (dP - D); dQ = scale * dS K; dK = scale * dS^T Q.
    """
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, H, N, d = Q.shape
    tau = _scale(d, scale)
    dQ, dK, dV = np.empty_like(Q), np.empty_like(K), np.empty_like(V)
    for b in range(B):
        for h in range(H):
            tok_mask = np.repeat(np.repeat(mask[b, h], block, axis=0), block, axis=1)
            s = np.where(tok_mask, tau * (Q[b, h] @ K[b, h].T), -np.inf)
            m = s.max(axis=1, keepdims=True)
            e = np.exp(s - m)
            P = e / e.sum(axis=1, keepdims=True)
            dV[b, h] = P.T @ dO[b, h]
            dP = dO[b, h] @ V[b, h].T
            D = (P * dP).sum(axis=1, keepdims=True)
            dS = P * (dP - D)
            dQ[b, h] = tau * (dS @ K[b, h])
            dK[b, h] = tau * (dS.T @ Q[b, h])
    return dQ, dK, dV


def _group_bwd(q, kk, vv, do, tau):
    s = tau * (q @ kk.T)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    P = e / e.sum(axis=1, keepdims=True)
    dP = do @ vv.T
    D = (P * dP).sum(axis=1, keepdims=True)
    dS = P * (dP - D)
    return tau * (dS @ kk), tau * (dS.T @ q), P.T @ do


def attn_bwd_groups(Q, K, V, dO, fwd_ptr, fwd_col, block: int, scale: Optional[float] = None):
    """Full dQ, dK, dV, evaluated group by group over the selected keys only.

    Same definition as attn_bwd_masked; each group's contribution to dK/dV
    is added into the key blocks of its list.
    """
    B, H, N, d = Q.shape
    G = N // block
    tau = _scale(d, scale)
    dQ = np.zeros((B, H, N, d))
    dK = np.zeros((B, H, N, d))
    dV = np.zeros((B, H, N, d))
    for b in range(B):
        for h in range(H):
            Kh, Vh = _f64(K[b, h]), _f64(V[b, h])
            for g in range(G):
                row = (b * H + h) * G + g
                cols = fwd_col[fwd_ptr[row]:fwd_ptr[row + 1]]
                keys = _group_keys(cols, block)
                sl = slice(g * block, (g + 1) * block)
                dq, dk, dv = _group_bwd(_f64(Q[b, h, sl]), Kh[keys], Vh[keys], _f64(dO[b, h, sl]), tau)
                dQ[b, h, sl] = dq
                dK[b, h, keys] += dk
                dV[b, h, keys] += dv
    return dQ, dK, dV


def attn_bwd_dq_rows(Q, K, V, dO, fwd_ptr, fwd_col, block: int, rows, scale: Optional[float] = None):
    """dQ of the listed groups (b, h, g), each from its own list only."""
    B, H, N, d = Q.shape
    G = N // block
    tau = _scale(d, scale)
    out = []
    for (b, h, g) in rows:
        row = (b * H + h) * G + g
        keys = _group_keys(fwd_col[fwd_ptr[row]:fwd_ptr[row + 1]], block)
        sl = slice(g * block, (g + 1) * block)
        dq, _, _ = _group_bwd(_f64(Q[b, h, sl]), _f64(K[b, h, keys]), _f64(V[b, h, keys]), _f64(dO[b, h, sl]), tau)
        out.append(dq)
    return out


def attn_bwd_kv_blocks(Q, K, V, dO, fwd_ptr, fwd_col, bwd_ptr, bwd_col, block: int, blocks,
                       scale: Optional[float] = None):
    """dK, dV of the listed key blocks (b, h, j).

    Sums the contribution of every group g in j's transposed list; each
    group's softmax is normalised over that group's whole list.
    """
    B, H, N, d = Q.shape
    G = N // block
    nb = N // block
    tau = _scale(d, scale)
    out = []
    for (b, h, j) in blocks:
        dk = np.zeros((block, d))
        dv = np.zeros((block, d))
        r = (b * H + h) * nb + j
        for g in bwd_col[bwd_ptr[r]:bwd_ptr[r + 1]]:
            g = int(g)
            row = (b * H + h) * G + g
            cols = np.asarray(fwd_col[fwd_ptr[row]:fwd_ptr[row + 1]])
            keys = _group_keys(cols, block)
            sl = slice(g * block, (g + 1) * block)
            _, dkk, dvv = _group_bwd(_f64(Q[b, h, sl]), _f64(K[b, h, keys]), _f64(V[b, h, keys]),
                                     _f64(dO[b, h, sl]), tau)
            pos = int(np.nonzero(cols == j)[0][0])
            dk += dkk[pos * block:(pos + 1) * block]
            dv += dvv[pos * block:(pos + 1) * block]
        out.append((dk, dv))
    return out


def attn_bwd_kv_blocks_given_stats(Q, K, V, dO, lse, D, bwd_ptr, bwd_col, block: int, blocks,
                                   scale: Optional[float] = None):
    """dK, dV of the listed key blocks (b, h, j), given each query row's
    softmax statistics: its log-sum-exp LSE_i over its whole list and
    D_i = sum_j P_ij dP_ij.

    With those two numbers the gradient of a key block needs only the tile of
    each group g in its transposed list: P = exp(scale * Q_g K_j^T - LSE_g),
    dP = dO_g V_j^T, dS = P * (dP - D_g), dV_j = sum_g P^T dO_g,
    dK_j = scale * sum_g dS^T Q_g -- the same closed form as attn_bwd_masked,
    restricted to the columns of block j.  It lets a block chosen by thousands
    of groups be checked without redoing each group's whole softmax; lse and
    D are [B, H, N] arrays (only the rows of the listed groups are read).
    """
    B, H, N, d = Q.shape
    nb = N // block
    tau = _scale(d, scale)
    out = []
    for (b, h, j) in blocks:
        ks = slice(j * block, (j + 1) * block)
        kj, vj = _f64(K[b, h, ks]), _f64(V[b, h, ks])
        dk = np.zeros((block, d))
        dv = np.zeros((block, d))
        r = (b * H + h) * nb + j
        for g in bwd_col[bwd_ptr[r]:bwd_ptr[r + 1]]:
            qs = slice(int(g) * block, (int(g) + 1) * block)
            q, do = _f64(Q[b, h, qs]), _f64(dO[b, h, qs])
            P = np.exp(tau * (q @ kj.T) - _f64(lse[b, h, qs])[:, None])
            dS = P * (do @ vj.T - _f64(D[b, h, qs])[:, None])
            dv += P.T @ do
            dk += tau * (dS.T @ q)
        out.append((dk, dv))
    return out


# --------------------------------------------------------------------------
# 3D cube query grouping ([nl] 2B, [hi] 2B: adjacent tokens in 3D space share
# their critical KV; queries are grouped in small cubes, e.g. 2x2x2)
# --------------------------------------------------------------------------

def cube_order(T: int, Hl: int, Wl: int, ct: int, cy: int, cx: int) -> np.ndarray:
    """perm[n_cube] = n_raster for the T x Hl x Wl latent grid cut into
    ct x cy x cx cubes.

    Raster order is n = (t*Hl + y)*Wl + x.  Cube order walks the cube grid
    (T/ct, Hl/cy, Wl/cx) in raster order and, inside each cube, its tokens in
    raster order (lt, ly, lx), so every run of ct*cy*cx consecutive positions
    is one cube: a query group / key block of the hot path becomes a cube.
    Written as the nested walk it is (small grids only).
    """
    if T % ct or Hl % cy or Wl % cx:
        raise ValueError("the cube must tile the grid")
    perm = []
    for bt in range(T // ct):
        for by in range(Hl // cy):
            for bx in range(Wl // cx):
                for lt in range(ct):
                    for ly in range(cy):
                        for lx in range(cx):
                            t, y, x = bt * ct + lt, by * cy + ly, bx * cx + lx
                            perm.append((t * Hl + y) * Wl + x)
    return np.asarray(perm, dtype=np.int64)


def permute_tokens(X, perm, inverse: bool = False) -> np.ndarray:
    """Token rows of X [B, H, N, d] into cube order (out[:, :, n] =
    X[:, :, perm[n]]) or, with inverse, back (out[:, :, perm[n]] = X[:, :, n]).
    Pure data movement: the dtype is kept."""
    X = np.asarray(X)
    perm = np.asarray(perm)
    if not inverse:
        return X[:, :, perm]
    out = np.empty_like(X)
    out[:, :, perm] = X
    return out


# --------------------------------------------------------------------------
# Mass-threshold selection ([nl] 2A and [hi] 2A: the critical KV pairs are
# those that carry about 90 % of the attention score)
# --------------------------------------------------------------------------

def mass_count_row(scores_row, tau: float, temperature: float, kmin: int, kmax: int) -> int:
    """m of one row: the predicted attention mass of block j is
    p_j = softmax(temperature * s)_j over the row; with the blocks in rank
    order (larger score first, equal scores by lower index), m is the
    smallest count whose leading blocks carry p-mass >= tau, clamped to
    [kmin, kmax].  A row holding a non-finite score gets m = kmax."""
    s = _f64(scores_row)
    if not np.all(np.isfinite(s)):
        return int(kmax)
    z = temperature * s
    p = np.exp(z - z.max())
    p = p / p.sum()
    cum = np.cumsum(p[_rank_order(s[None, :])[0]])
    m = min(int(np.searchsorted(cum, tau, side="left")) + 1, s.shape[0])
    return int(min(max(m, kmin), kmax))


def mass_lists(S, tau: float, temperature: float, kmin: int, kmax: int) -> Tuple[np.ndarray, np.ndarray]:
    """Forward CSR over all rows (b, h, g) of the mass-threshold selection:
    row (b, h, g) keeps the top mass_count_row(...) blocks, ascending."""
    S = _f64(S)
    B, H, G, nb = S.shape
    ptr = [0]
    cols = []
    for b in range(B):
        for h in range(H):
            for g in range(G):
                m = mass_count_row(S[b, h, g], tau, temperature, kmin, kmax)
                cols.append(topk_row(S[b, h, g], m))
                ptr.append(ptr[-1] + m)
    return np.asarray(ptr, dtype=np.int64), (np.concatenate(cols).astype(np.int64) if cols else np.zeros(0, np.int64))
