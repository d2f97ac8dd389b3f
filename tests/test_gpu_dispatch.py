"""The OP dispatcher on the GPU path (needs a GB300): heads the dispatcher
routes dense run the same kernels with every block selected (k = nb, the
fused call's select-all path), heads routed sparse keep their top-k lists;
both are checked against the fp64 oracle -- a dense head against plain dense
softmax attention (the oracle with every block in every list)."""
import numpy as np
import pytest
import torch

import oracle
from dynamic_block_sparse_projection_gb300 import workloads as wl
from parity_util import GRAD_REL_L2, O_MAX_ABS, O_REL_L2, SMALL, max_abs_beyond_rounding, rel_l2, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dynamic_block_sparse_projection_gb300 import binding
    return binding


def test_dense_routed_head_matches_dense_attention(dsv):
    w = SMALL["stress_small"]                      # 3 heads, per-head keep ratios
    x = wl.make_inputs(w, device="cuda")
    nb = w.nb
    # kept fractions 2/15, 12/15, 4/15 and a profile crossing 1 at rho = 0.5:
    # head 1 goes dense, heads 0 and 2 stay sparse
    ks = [2, 12, 4]
    k_out, dense = dsv.dispatch_heads(ks, nb, [0.1, 0.5, 1.0], [0.4, 1.0, 1.1])
    assert dense == [False, True, False] and k_out == [2, nb, 4]
    fp, fc, bp, bc = dsv.predict_topk_blocks(x.Q, x.K, x.Wq, x.Wk, k_out, w.block)
    O, lse = dsv.sparse_attn_fwd(x.Q, x.K, x.V, fp, fc, w.block)
    dQ, dK, dV = dsv.sparse_attn_bwd(x.Q, x.K, x.V, O, x.dO, lse, fp, fc, bp, bc, w.block)
    torch.cuda.synchronize()
    assert dsv.device_error()[0] == 0
    fpn, fcn = fp.cpu().numpy().astype(np.int64), fc.cpu().numpy().astype(np.int64)
    G = nb
    for b in range(w.B):
        for h in range(w.H):
            bh = b * w.H + h
            p = fpn[bh * G:(bh + 1) * G + 1]
            hp, hc = p - p[0], fcn[p[0]:p[-1]]
            if dense[h]:
                assert np.array_equal(hc, np.tile(np.arange(nb), G))   # every block, in order
            Q, K, V, dO = (to64(t[b:b + 1, h:h + 1]) for t in (x.Q, x.K, x.V, x.dO))
            if dense[h]:
                # plain dense softmax attention: the masked oracle with nothing masked
                mask = np.ones((1, 1, G, nb), dtype=bool)
                O_ref, _ = oracle.attn_fwd_masked(Q, K, V, mask, w.block)
                grads_ref = oracle.attn_bwd_masked(Q, K, V, dO, mask, w.block)
            else:
                O_ref, _ = oracle.attn_fwd_groups(Q, K, V, hp, hc, w.block)
                grads_ref = oracle.attn_bwd_groups(Q, K, V, dO, hp, hc, w.block)
            o = to64(O[b:b + 1, h:h + 1])
            assert rel_l2(o, O_ref) <= O_REL_L2 and max_abs_beyond_rounding(o, O_ref) <= O_MAX_ABS, (b, h, dense[h])
            for got, ref in zip((dQ, dK, dV), grads_ref):
                assert rel_l2(to64(got[b:b + 1, h:h + 1]), ref) <= GRAD_REL_L2, (b, h, dense[h])
