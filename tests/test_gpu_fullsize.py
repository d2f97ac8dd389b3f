"""GPU parity at the full workload sizes, on sampled outputs (needs a GB300).

The whole hot path runs at the benchmark's sizes and launch configuration;
the fp64 oracle then checks what it can evaluate one item at a time:

  scores    rows S[b,h,g,:] of sampled groups against the oracle's per-row form
  lists     every forward row bit-exact against the oracle's top-k fed the
            GPU's own fp32 scores (long518k: 64 rows per sampled head); for
            sampled heads the whole transposed CSR equal to the oracle's
            transpose of the GPU lists
  forward   O and lse of 16 sampled groups in each of 4 sampled heads against
            the per-group oracle
  backward  dQ of the same groups and dK/dV of up to 8 sampled key blocks per
            head (the least selected, the most selected with at most
            MAX_GROUPS groups, random ones) against the per-group / per-block
            oracle forms, on the GPU lists
  long lists  in the first sampled head, dK/dV of the key blocks with long
            transposed lists: against the per-block oracle (which redoes the
            whole softmax of every group in the list) a block of about the
            mean list length, the longest list within FULL_BUDGET group-blocks
            and, on latent123k_global, the head's least-chosen amplified global
            block; against the oracle's block form fed each row's LSE and
            D = rowsum(dO * O) from the GPU forward (those are checked against
            the oracle on the sampled groups) the most-selected block (3865
            groups at long518k), the most-selected global block and a
            90th-percentile block

The oracle sees one (b, h) slice at a time, as fp32 copies of the bf16 inputs
(exact), with the CSR rows of that slice re-based to (0, 0).
"""
import numpy as np
import pytest
import torch

import oracle
from dynamic_block_sparse_projection_gb300 import workloads as wl
from parity_util import (GRAD_REL_L2, LSE_MAX_ABS, O_MAX_ABS, O_REL_L2, SCORE_REL, max_abs_beyond_rounding,
                         rel_l2, score_err)

pytestmark = pytest.mark.gpu

FULL = ["latent16k", "latent123k_global", "stress61k", "long518k"]
MAX_GROUPS = 48
FULL_BUDGET = 45000       # groups x their list lengths the per-block oracle may redo for one block


@pytest.fixture(scope="module")
def dsv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dynamic_block_sparse_projection_gb300 import binding
    return binding


def _head_csr(ptr, col, bh, G):
    """CSR rows of one (b, h) slice, re-based so that the slice is (0, 0)."""
    p = ptr[bh * G:(bh + 1) * G + 1]
    return p - p[0], col[p[0]:p[-1]]


def _f32(t):
    return t.detach().float().cpu().numpy()[None, None]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_parity(dsv, name):
    w = wl.WORKLOADS[name]
    G = w.nb
    x = wl.make_inputs(w, device="cuda")
    S = dsv.predict_scores(x.Q, x.K, x.Wq, x.Wk, w.block)
    fp, fc, bp, bc = dsv.topk_blocks(S, x.k_per_head, w.block, w.N, w.d)
    O, lse = dsv.sparse_attn_fwd(x.Q, x.K, x.V, fp, fc, w.block)
    dQ, dK, dV = dsv.sparse_attn_bwd(x.Q, x.K, x.V, O, x.dO, lse, fp, fc, bp, bc, w.block)
    torch.cuda.synchronize()
    assert dsv.device_error()[0] == 0
    assert int(fp[-1]) == sum(x.k_per_head[h] for h in range(w.H)) * w.B * G

    fpn, fcn = fp.cpu().numpy().astype(np.int64), fc.cpu().numpy().astype(np.int64)
    bpn, bcn = bp.cpu().numpy().astype(np.int64), bc.cpu().numpy().astype(np.int64)
    rng = np.random.default_rng(97 + w.seed)
    heads = {(0, 0), (w.B - 1, w.H - 1)}
    while len(heads) < min(4, w.B * w.H):
        heads.add((int(rng.integers(w.B)), int(rng.integers(w.H))))
    heads = sorted(heads)
    checked = {"O": [], "dQ": [], "dK": [], "dV": []}

    # lists bit-exact on every row of the smaller workloads (a sample of rows at long518k)
    if w.B * w.H * G * G <= 64 << 20:
        Sn = S.cpu().numpy()
        for b in range(w.B):
            for h in range(w.H):
                hp_, hc_ = _head_csr(fpn, fcn, b * w.H + h, G)
                ref = oracle.topk_lists(Sn[b:b + 1, h:h + 1], [x.k_per_head[h]])
                assert np.array_equal(hp_, ref[0]) and np.array_equal(hc_, ref[1]), f"lists {name} head {(b, h)}"
    for (b, h) in heads:
        bh = b * w.H + h
        Qh, Kh, Vh, dOh = (_f32(t[b, h]) for t in (x.Q, x.K, x.V, x.dO))
        Wq, Wk = x.Wq[h:h + 1].double().cpu().numpy(), x.Wk[h:h + 1].double().cpu().numpy()
        groups = sorted({0, G - 1} | {int(v) for v in rng.integers(G, size=14)})
        hp, hc = _head_csr(fpn, fcn, bh, G)

        # scores: sampled rows
        ref = oracle.predict_scores_rows(Qh, Kh, Wq, Wk, w.block, [(0, 0, g) for g in groups])
        got = S[b, h, groups].double().cpu().numpy()
        assert score_err(got, ref) <= SCORE_REL, f"scores {name} head {(b, h)}"

        # forward lists: the oracle's top-k on the GPU's scores of the same rows
        k = int(x.k_per_head[h])
        rows_gpu = S[b, h].double().cpu().numpy()
        for g in list(groups) + [int(v) for v in rng.integers(G, size=64)]:
            assert np.array_equal(hc[hp[g]:hp[g + 1]], oracle.topk_row(rows_gpu[g], k)), (name, b, h, g)

        # transposed CSR of the head: the oracle's transpose of the GPU lists
        tp, tc = oracle.transpose_lists(hp, hc, 1, 1, G, G)
        gp, gc = _head_csr(bpn, bcn, bh, G)
        assert np.array_equal(tp, gp) and np.array_equal(tc, gc), f"transposed lists {name} head {(b, h)}"

        # forward: sampled groups
        for g, (o_ref, l_ref) in zip(groups, oracle.attn_fwd_groups(Qh, Kh, Vh, hp, hc, w.block,
                                                                     rows=[(0, 0, g) for g in groups])):
            sl = slice(g * w.block, (g + 1) * w.block)
            o = O[b, h, sl].double().cpu().numpy()
            checked["O"].append((o, o_ref))
            assert max_abs_beyond_rounding(o, o_ref) <= O_MAX_ABS
            assert np.max(np.abs(lse[b, h, sl].double().cpu().numpy() - l_ref)) <= LSE_MAX_ABS

        # backward: dQ of sampled groups (rel-L2 over all checked elements, below)
        for g, dq_ref in zip(groups, oracle.attn_bwd_dq_rows(Qh, Kh, Vh, dOh, hp, hc, w.block,
                                                              [(0, 0, g) for g in groups])):
            sl = slice(g * w.block, (g + 1) * w.block)
            checked["dQ"].append((dQ[b, h, sl].double().cpu().numpy(), dq_ref))

        # backward: dK, dV of sampled key blocks.  The per-block oracle redoes
        # the whole softmax of every group in the block's list, so only blocks
        # with at most MAX_GROUPS groups are sampled (the least selected, the
        # most selected among those, a random one); the gradient sums below
        # cover every block.
        lens = np.diff(gp)
        cheap = np.nonzero((lens > 0) & (lens <= MAX_GROUPS))[0]
        blocks = {int(np.argmin(lens))}
        if cheap.size:
            blocks |= {int(cheap[np.argmax(lens[cheap])])} | {int(v) for v in rng.choice(cheap, size=6)}
        blocks = sorted(blocks)
        for j, (dk_ref, dv_ref) in zip(blocks, oracle.attn_bwd_kv_blocks(Qh, Kh, Vh, dOh, hp, hc, gp, gc, w.block,
                                                                          [(0, 0, j) for j in blocks])):
            sl = slice(j * w.block, (j + 1) * w.block)
            dk = dK[b, h, sl].double().cpu().numpy()
            dv = dV[b, h, sl].double().cpu().numpy()
            if lens[j] == 0:
                assert np.all(dk == 0) and np.all(dv == 0)
            else:
                checked["dK"].append((dk, dk_ref))
                checked["dV"].append((dv, dv_ref))

        # gradient sums over every key of the head: each query's softmax row sums
        # to one, so sum_keys dV = sum_queries dO and sum_keys dK = 0 (every
        # query group has a non-empty list here)
        dKs = dK[b, h].double().sum(dim=0)
        assert torch.all(dKs.abs() <= 2e-2 * dK[b, h].double().abs().sum(dim=0) + 1e-3)
        assert rel_l2(dV[b, h].double().sum(dim=0).cpu().numpy(), x.dO[b, h].double().sum(dim=0).cpu().numpy()) <= 1e-2

    # long transposed lists, first sampled head
    b, h = heads[0]
    bh = b * w.H + h
    hp, hc = _head_csr(fpn, fcn, bh, G)
    gp, gc = _head_csr(bpn, bcn, bh, G)
    lens = np.diff(gp)
    row_len = np.diff(hp)
    cost = np.array([int(row_len[gc[gp[j]:gp[j + 1]]].sum()) for j in range(G)])   # group-blocks redone per block
    full_blocks = {"mean-length": int(np.argmin(np.abs(lens - lens.mean()) + 1e9 * (cost > FULL_BUDGET)))}
    within = np.nonzero(cost <= FULL_BUDGET)[0]
    full_blocks["longest within budget"] = int(within[np.argmax(lens[within])])
    stat_blocks = {"most-selected": int(np.argmax(lens)),
                   "90th percentile": int(np.argmin(np.abs(lens - np.percentile(lens, 90))))}
    if x.global_blocks and x.global_blocks[h]:
        gl = sorted(x.global_blocks[h], key=lambda j: lens[j])
        if cost[gl[0]] <= FULL_BUDGET:
            full_blocks["global, least chosen"] = gl[0]
        stat_blocks["global, most chosen"] = gl[-1]
    Qh, Kh, Vh, dOh = (_f32(t[b, h]) for t in (x.Q, x.K, x.V, x.dO))
    lse_h = lse[b, h].double().cpu().numpy()[None, None]
    D_h = (O[b, h].double() * x.dO[b, h].double()).sum(dim=-1).cpu().numpy()[None, None]
    for form, chosen in (("per-block oracle", full_blocks), ("block form given GPU LSE and D", stat_blocks)):
        js = list(chosen.values())
        if form == "per-block oracle":
            refs = oracle.attn_bwd_kv_blocks(Qh, Kh, Vh, dOh, hp, hc, gp, gc, w.block, [(0, 0, j) for j in js])
        else:
            refs = oracle.attn_bwd_kv_blocks_given_stats(Qh, Kh, Vh, dOh, lse_h, D_h, gp, gc, w.block,
                                                         [(0, 0, j) for j in js])
        for (what, j), (dk_ref, dv_ref) in zip(chosen.items(), refs):
            sl = slice(j * w.block, (j + 1) * w.block)
            ek = rel_l2(dK[b, h, sl].double().cpu().numpy(), dk_ref)
            ev = rel_l2(dV[b, h, sl].double().cpu().numpy(), dv_ref)
            print(f"{name} head {(b, h)} block {j} ({what}, {int(lens[j])} groups, {form}): "
                  f"dK rel-L2 {ek:.4f}, dV rel-L2 {ev:.4f}")
            assert ek <= GRAD_REL_L2 and ev <= GRAD_REL_L2, (name, what, j, ek, ev)

    # O max-abs: raw, and beyond the half-ulp rounding of the bf16 output
    raw = max(float(np.max(np.abs(a - r))) for a, r in checked["O"])
    beyond = max(max_abs_beyond_rounding(a, r) for a, r in checked["O"])
    print(f"{name} O max-abs: raw {raw:.4f}, beyond bf16 rounding {beyond:.4f}")

    # rel-L2 over all checked elements of the workload (the gate's definition)
    for nm, bar in (("O", O_REL_L2), ("dQ", GRAD_REL_L2), ("dK", GRAD_REL_L2), ("dV", GRAD_REL_L2)):
        got = np.concatenate([a.ravel() for a, _ in checked[nm]])
        ref = np.concatenate([r.ravel() for _, r in checked[nm]])
        e = rel_l2(got, ref)
        worst = max(rel_l2(a, r) for a, r in checked[nm])
        print(f"{name} {nm}: rel-L2 {e:.4f} over {len(checked[nm])} tiles (worst tile {worst:.4f})")
        assert e <= bar, f"{nm} {name}: rel-L2 {e:.4f} over {len(checked[nm])} tiles"

