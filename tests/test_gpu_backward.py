"""GPU parity of the sparse attention backward (needs a GB300).

dQ, dK, dV from the CUDA path (its own forward O and lse, then the backward)
against the fp64 oracle's closed-form gradient on the same lists:
rel-L2 <= 2e-2 each.  Also: blocks nobody selected get exactly zero, the
gradients obey the invariants of softmax attention, and runs are bitwise
repeatable.
"""
import numpy as np
import pytest
import torch

import oracle
from dynamic_block_sparse_projection_gb300 import workloads as wl
from parity_util import GRAD_REL_L2, SMALL, csr_to_device, oracle_lists, random_lists, rel_l2, to64

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


def _gpu_fwd_bwd(dsv, Q, K, V, dO, lists, block, scale=0.0):
    fp, fc, bp, bc = csr_to_device(lists, Q.device)
    O, lse = dsv.sparse_attn_fwd(Q, K, V, fp, fc, block, scale)
    dQ, dK, dV = dsv.sparse_attn_bwd(Q, K, V, O, dO, lse, fp, fc, bp, bc, block, scale)
    torch.cuda.synchronize()
    assert dsv.device_error()[0] == 0
    return O, lse, dQ, dK, dV


@pytest.mark.parametrize("name", CASES)
def test_backward_matches_oracle(dsv, name):
    w = _workload(name)
    x = wl.make_inputs(w, device="cuda")
    Q, K, V, dO = (to64(t) for t in (x.Q, x.K, x.V, x.dO))
    S_ref = oracle.predict_scores(Q, K, to64(x.Wq), to64(x.Wk), w.block)
    lists = oracle_lists(S_ref, x.k_per_head, w.nb)
    _, _, dQ, dK, dV = _gpu_fwd_bwd(dsv, x.Q, x.K, x.V, x.dO, lists, w.block)
    rQ, rK, rV = oracle.attn_bwd_groups(Q, K, V, dO, lists[0], lists[1], w.block)
    for got, ref, nm in ((dQ, rQ, "dQ"), (dK, rK, "dK"), (dV, rV, "dV")):
        e = rel_l2(to64(got), ref)
        assert e <= GRAD_REL_L2, f"{nm} rel-L2 {e:.3e}"
    # blocks that no group selected: exactly zero
    empty = np.nonzero(np.diff(lists[2]) == 0)[0]
    dKn, dVn = to64(dK), to64(dV)
    for r in empty:
        bh, j = divmod(int(r), w.nb)
        b, h = divmod(bh, w.H)
        assert np.all(dKn[b, h, j * w.block:(j + 1) * w.block] == 0)
        assert np.all(dVn[b, h, j * w.block:(j + 1) * w.block] == 0)


@pytest.mark.parametrize("block,d", [(64, 64), (64, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("k", [1, 3, "all"])
def test_backward_all_tile_shapes(dsv, block, d, k):
    rng = np.random.default_rng(block * 7 + d + (0 if k == "all" else k))
    B, H, G = 1, 2, 5
    N = G * block
    kk = G if k == "all" else k
    g = torch.Generator(device="cuda").manual_seed(11)
    Qb, Kb, Vb, dOb = (torch.randn(B, H, N, d, generator=g, device="cuda").to(torch.bfloat16) * 1.5 for _ in range(4))
    lists = random_lists(rng, B, H, G, [kk, kk])
    _, _, dQ, dK, dV = _gpu_fwd_bwd(dsv, Qb, Kb, Vb, dOb, lists, block, 0.11)
    rQ, rK, rV = oracle.attn_bwd_groups(to64(Qb), to64(Kb), to64(Vb), to64(dOb), lists[0], lists[1], block, 0.11)
    for got, ref in ((dQ, rQ), (dK, rK), (dV, rV)):
        assert rel_l2(to64(got), ref) <= GRAD_REL_L2


def test_backward_invariants_and_determinism(dsv):
    w = SMALL["global_small"]
    x = wl.make_inputs(w, device="cuda")
    S_ref = oracle.predict_scores(to64(x.Q), to64(x.K), to64(x.Wq), to64(x.Wk), w.block)
    lists = oracle_lists(S_ref, x.k_per_head, w.nb)
    a = _gpu_fwd_bwd(dsv, x.Q, x.K, x.V, x.dO, lists, w.block)
    b = _gpu_fwd_bwd(dsv, x.Q, x.K, x.V, x.dO, lists, w.block)
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    _, _, dQ, dK, dV = a
    dKs = dK.double().sum(dim=2)
    mag = dK.double().abs().sum(dim=2)
    assert torch.all(dKs.abs() <= 2e-2 * mag + 1e-3)
    dVs = dV.double().sum(dim=2)
    dOs = x.dO.double().sum(dim=2)
    assert rel_l2(dVs.cpu().numpy(), dOs.cpu().numpy()) <= 1e-2


def test_backward_empty_group_list(dsv):
    B, H, N, d, block = 1, 1, 256, 128, 64
    g = torch.Generator(device="cuda").manual_seed(13)
    Qb, Kb, Vb, dOb = (torch.randn(B, H, N, d, generator=g, device="cuda").to(torch.bfloat16) for _ in range(4))
    fp_ = np.array([0, 2, 2, 3, 4])
    fc_ = np.array([1, 3, 0, 2])
    bp_, bc_ = oracle.transpose_lists(fp_, fc_, B, H, 4, 4)
    _, _, dQ, dK, dV = _gpu_fwd_bwd(dsv, Qb, Kb, Vb, dOb, (fp_, fc_, bp_, bc_), block)
    assert torch.all(dQ[0, 0, 64:128] == 0)
    # the oracle's per-group and per-block forms never visit the empty group
    args = (to64(Qb), to64(Kb), to64(Vb), to64(dOb), fp_, fc_)
    rows = [(0, 0, 0), (0, 0, 2), (0, 0, 3)]
    for (_, _, gg), ref in zip(rows, oracle.attn_bwd_dq_rows(*args, block, rows)):
        sl = slice(gg * 64, (gg + 1) * 64)
        assert rel_l2(to64(dQ)[0, 0, sl], ref) <= GRAD_REL_L2
    blocks = [(0, 0, j) for j in range(4)]
    for (_, _, j), (rk, rv) in zip(blocks, oracle.attn_bwd_kv_blocks(*args, bp_, bc_, block, blocks)):
        sl = slice(j * 64, (j + 1) * 64)
        assert rel_l2(to64(dK)[0, 0, sl], rk) <= GRAD_REL_L2
        assert rel_l2(to64(dV)[0, 0, sl], rv) <= GRAD_REL_L2


def test_backward_stages_equal_single_call(dsv):
    """preprocess, dK/dV and dQ run as separate calls (dQ first) give the
    single call's gradients bit for bit."""
    w = SMALL["stress_small"]
    x = wl.make_inputs(w, device="cuda")
    S_ref = oracle.predict_scores(to64(x.Q), to64(x.K), to64(x.Wq), to64(x.Wk), w.block)
    lists = oracle_lists(S_ref, x.k_per_head, w.nb)
    O, lse, dQ, dK, dV = _gpu_fwd_bwd(dsv, x.Q, x.K, x.V, x.dO, lists, w.block)
    fp, fc, bp, bc = csr_to_device(lists, x.Q.device)
    B, H, N, d = x.Q.shape
    nbytes = dsv.attn_bwd_workspace_bytes(B, H, N, d, w.block)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    sQ, sK, sV = (torch.full_like(x.Q, 7.0) for _ in range(3))
    dsv.attn_bwd_preprocess(O, x.dO, lse, w.block, workspace=ws)
    dsv.attn_bwd_dq(x.Q, x.K, x.V, x.dO, fp, fc, w.block, out=sQ, workspace=ws)
    dsv.attn_bwd_dkdv(x.Q, x.K, x.V, x.dO, bp, bc, w.block, outs=(sK, sV), workspace=ws)
    torch.cuda.synchronize()
    assert dsv.device_error()[0] == 0
    assert torch.equal(sQ, dQ) and torch.equal(sK, dK) and torch.equal(sV, dV)

