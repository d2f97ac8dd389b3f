"""Failure detection on the GPU, without a fault (needs a GB300).

The kernels record what they detect in a per-device error word instead of
trapping:
  * an out-of-range block index in a caller's CSR list: DSV_ERR_BAD_INDEX,
    with the row as info; the kernel clamps the index before any load, so
    nothing outside the tensors is read;
  * a wait that runs past its time limit: DSV_ERR_TIMEOUT, with the wait's
    id as info; the kernel gives up and returns.  The time-out is made by
    the library's self-test kernel, whose only wait is on a barrier that
    nothing arrives at, under a short limit.
Each test then clears the word, restores the default limit and runs the tiny
hot path again, checking it against the fp64 oracle: the context stays usable.
"""
import numpy as np
import pytest
import torch

import oracle
from dynamic_block_sparse_projection_gb300 import workloads as wl
from parity_util import O_REL_L2, GRAD_REL_L2, rel_l2, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dynamic_block_sparse_projection_gb300 import binding
    return binding


def _tiny_path_matches_oracle(dsv):
    w = wl.WORKLOADS["tiny"]
    x = wl.make_inputs(w, device="cuda")
    S = dsv.predict_scores(x.Q, x.K, x.Wq, x.Wk, w.block)
    fp, fc, bp, bc = dsv.topk_blocks(S, x.k_per_head, w.block, w.N, w.d)
    O, lse = dsv.sparse_attn_fwd(x.Q, x.K, x.V, fp, fc, w.block)
    dQ, dK, dV = dsv.sparse_attn_bwd(x.Q, x.K, x.V, O, x.dO, lse, fp, fc, bp, bc, w.block)
    st, info = dsv.device_error()
    assert st == dsv.DSV_OK, (dsv.status_string(st), info)
    Q, K, V, dO = (to64(t) for t in (x.Q, x.K, x.V, x.dO))
    rfp, rfc = oracle.topk_lists(to64(S), x.k_per_head)
    assert np.array_equal(fc.cpu().numpy(), rfc)
    O_ref, _ = oracle.attn_fwd_groups(Q, K, V, rfp, rfc, w.block)
    assert rel_l2(to64(O), O_ref) <= O_REL_L2
    for got, ref in zip((dQ, dK, dV), oracle.attn_bwd_groups(Q, K, V, dO, rfp, rfc, w.block)):
        assert rel_l2(to64(got), ref) <= GRAD_REL_L2


def test_out_of_range_index_is_reported_and_the_context_recovers(dsv):
    w = wl.WORKLOADS["tiny"]
    x = wl.make_inputs(w, device="cuda")
    dsv.clear_device_error()
    S = dsv.predict_scores(x.Q, x.K, x.Wq, x.Wk, w.block)
    fp, fc, _, _ = dsv.topk_blocks(S, x.k_per_head, w.block, w.N, w.d)
    bad_row = 3                                    # (b, h, g) = (0, 0, 3)
    fc_bad = fc.clone()
    fc_bad[int(fp[bad_row])] = w.nb                # one past the last key block
    dsv.sparse_attn_fwd(x.Q, x.K, x.V, fp, fc_bad, w.block)
    st, info = dsv.device_error()
    assert st == dsv.DSV_ERR_BAD_INDEX, dsv.status_string(st)
    assert info == bad_row
    dsv.clear_device_error()
    assert dsv.device_error()[0] == dsv.DSV_OK
    _tiny_path_matches_oracle(dsv)


def test_wait_time_out_is_reported_and_the_context_recovers(dsv):
    dsv.clear_device_error()
    try:
        dsv.set_wait_limit_ns(20_000_000)          # 20 ms
        dsv.selftest_wait_timeout()
        st, info = dsv.device_error()
    finally:
        dsv.set_wait_limit_ns(0)                   # the default limit again
    assert st == dsv.DSV_ERR_TIMEOUT, dsv.status_string(st)
    assert info == dsv.SELFTEST_WAIT_ID
    dsv.clear_device_error()
    assert dsv.device_error()[0] == dsv.DSV_OK
    _tiny_path_matches_oracle(dsv)


def test_first_error_wins(dsv):
    """The word keeps the first error: a later time-out does not overwrite an
    out-of-range index, and a clear resets it."""
    w = wl.WORKLOADS["tiny"]
    x = wl.make_inputs(w, device="cuda")
    dsv.clear_device_error()
    S = dsv.predict_scores(x.Q, x.K, x.Wq, x.Wk, w.block)
    fp, fc, _, _ = dsv.topk_blocks(S, x.k_per_head, w.block, w.N, w.d)
    fc_bad = fc.clone()
    fc_bad[0] = -1
    dsv.sparse_attn_fwd(x.Q, x.K, x.V, fp, fc_bad, w.block)
    try:
        dsv.set_wait_limit_ns(5_000_000)
        dsv.selftest_wait_timeout()
        st, info = dsv.device_error()
    finally:
        dsv.set_wait_limit_ns(0)
    assert st == dsv.DSV_ERR_BAD_INDEX and info == 0
    dsv.clear_device_error()
    _tiny_path_matches_oracle(dsv)
