"""GPU parity of the fused predictor + top-k, dsv_predict_topk_blocks (needs a GB300).

The fused call never stores the score matrix; for checking it can write the
scores its selection used.  Against the fp64 oracle, on the same seeded inputs:
  * those scores: |dS| <= 1e-4 * max(|S_ref|, row rms) against
    oracle.predict_scores (the tf32 hi/lo products stay near 1e-6);
  * the lists: bit-exact against the oracle's top-k of those same fp32 scores
    (an integer decision taken on the same keys), and the transposed lists
    against the oracle's transpose;
  * the cases that take the exact fallback inside the kernel (rows of equal
    scores, many exact ties), k = 1 and k = nb, and bitwise repeatability;
  * at full size, sampled score rows and every list row (sampled rows at
    long518k), with the two-call path's lists compared for information.
"""
import numpy as np
import pytest
import torch

import oracle
from dynamic_block_sparse_projection_gb300 import workloads as wl
from parity_util import SCORE_REL, SMALL, oracle_lists, score_err, to64

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


def _fused(dsv, x, w, ks=None):
    G = w.nb
    S = torch.full((w.B, w.H, G, G), float("nan"), dtype=torch.float32, device="cuda")
    lists = dsv.predict_topk_blocks(x.Q, x.K, x.Wq, x.Wk, ks or x.k_per_head, w.block, scores=S)
    torch.cuda.synchronize()
    st, info = dsv.device_error()
    assert st == dsv.DSV_OK, (dsv.status_string(st), info)
    return S, lists


def _check_lists_exact(S, lists, ks, G):
    S64 = to64(S)
    rfp, rfc, rbp, rbc = oracle_lists(S64, ks, G)
    fp, fc, bp, bc = (t.cpu().numpy() for t in lists)
    assert np.array_equal(fp, rfp)
    assert np.array_equal(fc, rfc)
    assert np.array_equal(bp, rbp)
    assert np.array_equal(bc, rbc)


@pytest.mark.parametrize("name", CASES)
def test_fused_scores_and_lists_match_oracle(dsv, name):
    w = _workload(name)
    x = wl.make_inputs(w, device="cuda", with_dO=False)
    S, lists = _fused(dsv, x, w)
    S_ref = oracle.predict_scores(to64(x.Q), to64(x.K), to64(x.Wq), to64(x.Wk), w.block)
    err = score_err(to64(S), S_ref)
    print(f"{name}: fused score error {err:.2e} of the gate's scale")
    assert err <= SCORE_REL
    _check_lists_exact(S, lists, x.k_per_head, w.nb)


@pytest.mark.parametrize("k", [1, "nb"])
def test_fused_k_extremes(dsv, k):
    w = SMALL["global_small"]
    x = wl.make_inputs(w, device="cuda", with_dO=False)
    ks = [w.nb if k == "nb" else 1] * w.H
    S, lists = _fused(dsv, x, w, ks)
    _check_lists_exact(S, lists, ks, w.nb)


def test_fused_equal_scores_take_the_exact_fallback(dsv):
    """Head 0's keys are one repeated row: every score of a row is equal (the
    whole row lands in one bin), so the kernel's exact radix select must keep
    the k lowest block indices; head 1 duplicates every other key block, so
    its rows hold many exact ties that the ranked threshold bin resolves to
    the lower index."""
    w = SMALL["global_small"]
    x = wl.make_inputs(w, device="cuda", with_dO=False)
    x.K[:, 0] = x.K[:, 0, :1].clone()
    Kb = x.K[:, 1].reshape(w.B, w.nb, w.block, w.d)            # a view of head 1
    assert Kb.data_ptr() == x.K[:, 1].data_ptr()
    Kb[:, 1::2] = Kb[:, 0:-1:2][:, : Kb[:, 1::2].shape[1]].clone()
    S, lists = _fused(dsv, x, w)
    S64 = to64(S)
    assert np.all(S64[:, 0] == S64[:, 0, :, :1])               # constant rows
    _check_lists_exact(S, lists, x.k_per_head, w.nb)
    fc = lists[1].cpu().numpy()
    k0 = x.k_per_head[0]
    assert np.array_equal(fc[:k0], np.arange(k0))             # first row of head 0: the lowest indices


def test_fused_bitwise_repeatable(dsv):
    w = SMALL["long_small"]
    x = wl.make_inputs(w, device="cuda", with_dO=False)
    S1, l1 = _fused(dsv, x, w)
    l1 = [t.clone() for t in l1]
    S2, l2 = _fused(dsv, x, w)
    assert torch.equal(S1, S2)
    for a, b in zip(l1, l2):
        assert torch.equal(a, b)


def test_fused_many_heads_split_launch(dsv):
    """Enough heads that the select kernel's items (128 groups of one head
    each) fill two or more waves of one CTA per SM with a partly filled wave
    left: that wave runs as a launch of its own while the transposed lists of
    the heads already selected are built on the second stream.  Every list,
    forward and transposed, must still match the oracle's top-k of the fused
    scores; G = 260 leaves a 4-group tile at the end of every head."""
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = 3                                                  # ceil(260 / 128)
    H = -(-2 * nsm // tiles) + 1
    while (H * tiles) % nsm == 0:
        H += 1
    w = wl.scaled(wl.WORKLOADS["latent16k"], name="many_heads", H=H, d=64, T=26, Hl=10, Wl=128)
    assert w.nb == 260 and H * tiles >= 2 * nsm
    x = wl.make_inputs(w, device="cuda", with_dO=False)
    S, lists = _fused(dsv, x, w)
    _check_lists_exact(S, lists, x.k_per_head, w.nb)


FULL = ["latent16k", "latent123k_global", "stress61k", "long518k"]


@pytest.mark.parametrize("name", FULL)
def test_fused_full_size(dsv, name):
    w = wl.WORKLOADS[name]
    G = w.nb
    x = wl.make_inputs(w, device="cuda", with_dO=False)
    S, lists = _fused(dsv, x, w)
    fp, fc, bp, bc = (t.cpu().numpy().astype(np.int64) for t in lists)
    assert int(fp[-1]) == sum(x.k_per_head) * w.B * G
    rng = np.random.default_rng(211 + w.seed)
    # scores: 16 sampled groups in each of 3 heads against the oracle's rows
    for bh in sorted({0, w.B * w.H - 1, int(rng.integers(w.B * w.H))}):
        b, h = divmod(bh, w.H)
        groups = sorted({0, G - 1} | {int(v) for v in rng.integers(G, size=14)})
        f = lambda t: t[b, h].float().cpu().numpy()[None, None]  # noqa: E731
        ref = oracle.predict_scores_rows(f(x.Q), f(x.K), x.Wq[h:h + 1].double().cpu().numpy(),
                                         x.Wk[h:h + 1].double().cpu().numpy(), w.block, [(0, 0, g) for g in groups])
        assert score_err(S[b, h, groups].double().cpu().numpy(), ref) <= SCORE_REL, (name, b, h)
    # lists: every row (sampled rows at long518k) bit-exact against the oracle's top-k of the fused scores
    two_call = dsv.topk_blocks(dsv.predict_scores(x.Q, x.K, x.Wq, x.Wk, w.block), x.k_per_head, w.block, w.N, w.d)
    fc2 = two_call[1].cpu().numpy()
    differ = 0
    for b in range(w.B):
        for h in range(w.H):
            k = x.k_per_head[h]
            bh = b * w.H + h
            Sh = S[b, h].double().cpu().numpy()
            rows = range(G) if G * G * w.B * w.H <= 64 << 20 else sorted({int(v) for v in rng.integers(G, size=48)})
            for g in rows:
                r0 = int(fp[bh * G + g])
                got = fc[r0:r0 + k]
                assert np.array_equal(got, oracle.topk_row(Sh[g], k)), (name, b, h, g)
                differ += int(not np.array_equal(got, fc2[r0:r0 + k]))
    # transposed lists of two heads: the oracle's transpose of the fused lists
    for bh in (0, w.B * w.H - 1):
        p = fp[bh * G:(bh + 1) * G + 1]
        tp, tc = oracle.transpose_lists(p - p[0], fc[p[0]:p[-1]], 1, 1, G, G)
        q = bp[bh * G:(bh + 1) * G + 1]
        assert np.array_equal(q - q[0], tp) and np.array_equal(bc[q[0]:q[-1]], tc)
    print(f"{name}: rows whose fused list differs from the two-call path's (near-ties of fp32 vs tf32x3 sums): "
          f"{differ}")
