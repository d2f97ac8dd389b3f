"""The Python binding's host side, run to the library call on the CPU.

The device check, the device guard, the stream lookup and the library are
replaced by stand-ins that record what they are given, so every wrapper runs
its argument handling end to end without a GPU: the right entry point is
called once, with the tensors' addresses, the shape the library needs, a
workspace of the size the library asked for, and outputs of the documented
shapes.  (The real calls run in the GPU tests.)
"""
import contextlib

import pytest
import torch


@pytest.fixture()
def fake(monkeypatch):
    from dynamic_block_sparse_projection_gb300.build import build
    build()
    from dynamic_block_sparse_projection_gb300 import binding

    calls = []

    class FakeLib:
        def __getattr__(self, name):
            if name.endswith("_workspace_bytes"):
                return lambda s: 4096 + s.B * s.H * s.N
            def fn(*args):
                calls.append((name, args))
                return 0
            return fn

    monkeypatch.setattr(binding, "lib", FakeLib())
    monkeypatch.setattr(binding, "_need", lambda *a, **k: None)
    monkeypatch.setattr(binding, "_stream", lambda dev, stream=None: 1234)
    monkeypatch.setattr(torch.cuda, "device", lambda dev: contextlib.nullcontext())
    return binding, calls


def _inputs(B=1, H=2, N=256, d=64, r=16):
    bf = torch.bfloat16
    Q, K, V, dO = (torch.zeros(B, H, N, d, dtype=bf) for _ in range(4))
    Wq, Wk = torch.zeros(H, d, r), torch.zeros(H, d, r)
    return Q, K, V, dO, Wq, Wk


def test_every_wrapper_reaches_its_entry_point(fake):
    dsv, calls = fake
    Q, K, V, dO, Wq, Wk = _inputs()
    B, H, N, d = Q.shape
    blk, G = 64, 4
    for fn, name in ((dsv.predict_scores, "dsv_predict_scores"), (dsv.predict_scores_max, "dsv_predict_scores_max")):
        S = fn(Q, K, Wq, Wk, blk)
        assert S.shape == (B, H, G, G) and S.dtype == torch.float32
        nm, args = calls[-1]
        assert nm == name and args[0] == Q.data_ptr() and args[3] == Wk.data_ptr()
        s = args[4]
        assert (s.B, s.H, s.N, s.d, s.block, s.r) == (B, H, N, d, blk, 16)
        assert args[7] == 4096 + B * H * N and args[8] == 1234
    lists = dsv.topk_blocks(S, [2, 3], blk, N, d)
    nnz = B * G * 5
    assert [t.numel() for t in lists] == [B * H * G + 1, nnz, B * H * G + 1, nnz]
    nm, args = calls[-1]
    assert nm == "dsv_topk_blocks" and list(args[2]) == [2, 3]
    outs = dsv.topk_mass_blocks(S, 0.9, blk, N, d, trim=False)
    nm, args = calls[-1]
    assert nm == "dsv_topk_mass_blocks" and args[4:6] == (1, G)
    assert abs(args[3] - 1 / 8.0) < 1e-12                        # temperature 1/sqrt(d)
    assert args[10] == B * H * G * G                             # column capacity
    dsv.topk_blocks_noalloc(S, [2, 3], blk, N, d, outs=lists)
    assert calls[-1][0] == "dsv_topk_blocks_noalloc"
    fp, fc, bp, bc = lists
    O, lse = dsv.sparse_attn_fwd(Q, K, V, fp, fc, blk)
    assert O.shape == Q.shape and lse.shape == (B, H, N) and calls[-1][0] == "dsv_sparse_attn_fwd"
    assert calls[-1][1][6] == 0.0                                # scale 0: the library's 1/sqrt(d)
    grads = dsv.sparse_attn_bwd(Q, K, V, O, dO, lse, fp, fc, bp, bc, blk, 0.25)
    assert [g.shape for g in grads] == [Q.shape] * 3 and calls[-1][0] == "dsv_sparse_attn_bwd"
    assert calls[-1][1][11] == 0.25
    ws = torch.empty(1000, dtype=torch.float32)
    dsv.attn_bwd_preprocess(O, dO, lse, blk, workspace=ws)
    assert calls[-1][0] == "dsv_attn_bwd_preprocess" and calls[-1][1][5] == 4000      # bytes, not elements
    dsv.attn_bwd_dkdv(Q, K, V, dO, bp, bc, blk, outs=grads[1:], workspace=ws)
    assert calls[-1][0] == "dsv_attn_bwd_dkdv" and calls[-1][1][11] == 4000
    dsv.attn_bwd_dq(Q, K, V, dO, fp, fc, blk, out=grads[0], workspace=ws)
    assert calls[-1][0] == "dsv_attn_bwd_dq" and calls[-1][1][10] == 4000
    y = dsv.cube_permute(Q, (4, 8, 8), (1, 8, 8), inverse=True)
    nm, args = calls[-1]
    assert nm == "dsv_cube_permute" and y.shape == Q.shape and args[3:10] == (4, 8, 8, 1, 8, 8, 1)


def test_caller_buffers_are_used_as_given(fake):
    dsv, calls = fake
    Q, K, V, dO, Wq, Wk = _inputs()
    S = torch.empty(1, 2, 4, 4)
    ws = torch.empty(1 << 16, dtype=torch.uint8)
    assert dsv.predict_scores(Q, K, Wq, Wk, 64, out=S, workspace=ws) is S
    assert calls[-1][1][5] == S.data_ptr() and calls[-1][1][6] == ws.data_ptr()
    with pytest.raises(ValueError, match="workspace needs"):
        dsv.predict_scores(Q, K, Wq, Wk, 64, workspace=torch.empty(16, dtype=torch.uint8))
    outs = tuple(torch.empty(n, dtype=torch.int32) for n in (9, 40, 9, 40))    # longer columns are fine
    got = dsv.topk_blocks(S, [2, 3], 64, 256, outs=outs)
    assert got[0] is outs[0] and got[1].numel() == 20 and got[1].data_ptr() == outs[1].data_ptr()
