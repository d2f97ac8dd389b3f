"""The C-ABI library: builds, loads, exports every declared symbol, and rejects
bad arguments on the host before any launch (CPU only; no compute calls)."""
import ctypes
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent


@pytest.fixture(scope="module")
def lib():
    from dynamic_block_sparse_projection_gb300.build import build
    build()
    from dynamic_block_sparse_projection_gb300 import binding
    return binding


def _declared():
    text = (ROOT / "include" / "dsv.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsv_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 12
    raw = ctypes.CDLL(str(lib._LIB_PATH))
    for n in names:
        assert hasattr(raw, n), n
    assert set(names) == set(lib.EXPORTS)


def test_status_strings_and_version(lib):
    assert lib.status_string(0) == "ok"
    assert "argument" in lib.status_string(1)
    assert lib.lib.dsv_version() >= 10000
    assert lib.status_string(99) == "unknown status"
    assert "consistency" in lib.status_string(lib.DSV_ERR_INTERNAL)


def _shape(lib, B=1, H=2, N=512, d=128, block=128, r=16):
    return lib.Shape(B, H, N, d, block, r)


def test_workspace_queries(lib):
    s = _shape(lib)
    G = 4
    assert lib.lib.dsv_predict_workspace_bytes(s) >= 2 * 1 * 2 * G * 16 * 4
    assert lib.lib.dsv_topk_workspace_bytes(s) >= 2 * G * 4
    assert lib.lib.dsv_attn_bwd_workspace_bytes(s) >= 1 * 2 * 512 * 4
    assert lib.lib.dsv_topk_workspace_bytes(_shape(lib, d=96)) == 0     # unsupported -> 0
    assert lib.lib.dsv_predict_workspace_bytes(_shape(lib, N=0)) == 0


FAKE = 1 << 20          # an aligned, never dereferenced address


def test_host_validation_predict(lib):
    L = lib.lib
    ws = L.dsv_predict_workspace_bytes(_shape(lib))
    ok = (FAKE, FAKE, FAKE, FAKE)
    assert L.dsv_predict_scores(*ok, _shape(lib, d=96), FAKE, FAKE, ws, None) == lib.DSV_ERR_UNSUPPORTED
    assert L.dsv_predict_scores(*ok, _shape(lib, block=32), FAKE, FAKE, ws, None) == lib.DSV_ERR_UNSUPPORTED
    assert L.dsv_predict_scores(*ok, _shape(lib, r=12), FAKE, FAKE, ws, None) == lib.DSV_ERR_UNSUPPORTED
    assert L.dsv_predict_scores(*ok, _shape(lib, N=500), FAKE, FAKE, ws, None) == lib.DSV_ERR_INVALID_ARG
    assert L.dsv_predict_scores(*ok, _shape(lib, B=-1), FAKE, FAKE, ws, None) == lib.DSV_ERR_INVALID_ARG
    assert L.dsv_predict_scores(None, FAKE, FAKE, FAKE, _shape(lib), FAKE, FAKE, ws, None) == lib.DSV_ERR_INVALID_ARG
    assert L.dsv_predict_scores(FAKE + 8, FAKE, FAKE, FAKE, _shape(lib), FAKE, FAKE, ws, None) == lib.DSV_ERR_INVALID_ARG
    assert L.dsv_predict_scores(*ok, _shape(lib), FAKE, FAKE + 16, ws, None) == lib.DSV_ERR_INVALID_ARG
    assert L.dsv_predict_scores(*ok, _shape(lib), FAKE, FAKE, ws - 1, None) == lib.DSV_ERR_INVALID_ARG
    # an empty problem is valid and launches nothing
    assert L.dsv_predict_scores(None, None, None, None, _shape(lib, N=0), None, None, 0, None) == lib.DSV_OK


def test_host_validation_topk(lib):
    L = lib.lib
    s = _shape(lib)
    ws = L.dsv_topk_workspace_bytes(s)
    k = (ctypes.c_int32 * 2)(2, 3)
    args = (FAKE, FAKE, FAKE, FAKE, FAKE, ws)
    assert L.dsv_topk_blocks(FAKE, s, (ctypes.c_int32 * 2)(0, 3), FAKE, *args, None) == lib.DSV_ERR_INVALID_ARG
    assert L.dsv_topk_blocks(FAKE, s, (ctypes.c_int32 * 2)(2, 5), FAKE, *args, None) == lib.DSV_ERR_INVALID_ARG
    assert L.dsv_topk_blocks(FAKE, s, None, FAKE, *args, None) == lib.DSV_ERR_INVALID_ARG
    assert L.dsv_topk_blocks(FAKE, s, k, FAKE, FAKE, FAKE, FAKE, FAKE, ws - 4, None) == lib.DSV_ERR_INVALID_ARG
    big = _shape(lib, N=128 * 8193, H=1)
    assert L.dsv_topk_blocks(FAKE, big, k, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40, None) == lib.DSV_ERR_UNSUPPORTED
    assert L.dsv_topk_blocks(FAKE, _shape(lib, H=1025), k, *((FAKE,) * 5), ws, None) == lib.DSV_ERR_UNSUPPORTED


def test_host_validation_attention(lib):
    L = lib.lib
    s = _shape(lib)
    assert L.dsv_sparse_attn_fwd(FAKE, FAKE, FAKE, s, FAKE, None, 0.0, FAKE, FAKE, None) == lib.DSV_ERR_INVALID_ARG
    assert L.dsv_sparse_attn_fwd(FAKE, FAKE, FAKE + 2, s, FAKE, FAKE, 0.0, FAKE, FAKE, None) == lib.DSV_ERR_INVALID_ARG
    assert L.dsv_sparse_attn_fwd(FAKE, FAKE, FAKE, _shape(lib, d=32), FAKE, FAKE, 0.0, FAKE, FAKE, None) == \
        lib.DSV_ERR_UNSUPPORTED
    ws = L.dsv_attn_bwd_workspace_bytes(s)
    p = (FAKE,) * 6
    assert L.dsv_sparse_attn_bwd(*p, s, FAKE, FAKE, FAKE, FAKE, 0.0, FAKE, FAKE, FAKE, FAKE, ws - 1, None) == \
        lib.DSV_ERR_INVALID_ARG
    assert L.dsv_sparse_attn_bwd(*p, s, FAKE, FAKE, None, FAKE, 0.0, FAKE, FAKE, FAKE, FAKE, ws, None) == \
        lib.DSV_ERR_INVALID_ARG
    assert L.dsv_sparse_attn_bwd(*p, s, FAKE, FAKE, FAKE, FAKE, 0.0, FAKE, FAKE, FAKE, FAKE + 64, ws, None) == \
        lib.DSV_ERR_INVALID_ARG


def test_host_validation_backward_stages(lib):
    L = lib.lib
    s = _shape(lib)
    ws = L.dsv_attn_bwd_workspace_bytes(s)
    assert L.dsv_attn_bwd_preprocess(FAKE, FAKE, FAKE, s, FAKE, ws - 1, None) == lib.DSV_ERR_INVALID_ARG
    assert L.dsv_attn_bwd_preprocess(FAKE, None, FAKE, s, FAKE, ws, None) == lib.DSV_ERR_INVALID_ARG
    assert L.dsv_attn_bwd_preprocess(FAKE, FAKE, FAKE, s, FAKE + 64, ws, None) == lib.DSV_ERR_INVALID_ARG
    assert L.dsv_attn_bwd_preprocess(FAKE, FAKE, FAKE, _shape(lib, d=96), FAKE, ws, None) == lib.DSV_ERR_UNSUPPORTED
    p4 = (FAKE,) * 4
    assert L.dsv_attn_bwd_dkdv(*p4, s, FAKE, None, 0.0, FAKE, FAKE, FAKE, ws, None) == lib.DSV_ERR_INVALID_ARG
    assert L.dsv_attn_bwd_dkdv(*p4, s, FAKE, FAKE, 0.0, FAKE + 2, FAKE, FAKE, ws, None) == lib.DSV_ERR_INVALID_ARG
    assert L.dsv_attn_bwd_dkdv(*p4, s, FAKE, FAKE, 0.0, FAKE, FAKE, FAKE, ws - 1, None) == lib.DSV_ERR_INVALID_ARG
    assert L.dsv_attn_bwd_dq(*p4, s, None, FAKE, 0.0, FAKE, FAKE, ws, None) == lib.DSV_ERR_INVALID_ARG
    assert L.dsv_attn_bwd_dq(*p4, s, FAKE, FAKE, 0.0, FAKE, FAKE + 64, ws, None) == lib.DSV_ERR_INVALID_ARG
    assert L.dsv_attn_bwd_dq(*p4, _shape(lib, N=500), FAKE, FAKE, 0.0, FAKE, FAKE, ws, None) == \
        lib.DSV_ERR_INVALID_ARG
    empty = _shape(lib, B=0)
    assert L.dsv_attn_bwd_dq(*p4, empty, None, None, 0.0, None, None, 0, None) == 0



def test_host_validation_cube_permute(lib):
    L = lib.lib
    s = _shape(lib, N=512, block=128)            # grid 2 x 16 x 16, cube 2 x 8 x 8
    grid, cube = (2, 16, 16), (2, 8, 8)
    far = FAKE + (64 << 20)                      # a second buffer that does not overlap the first
    assert L.dsv_cube_permute(FAKE, far, s, 2, 16, 16, 1, 8, 8, 0, None) == lib.DSV_ERR_INVALID_ARG   # volume != block
    assert L.dsv_cube_permute(FAKE, far, s, 2, 16, 17, *cube, 0, None) == lib.DSV_ERR_INVALID_ARG     # T*Hl*Wl != N
    assert L.dsv_cube_permute(FAKE, far, _shape(lib, N=384), 2, 12, 16, *cube, 0, None) == \
        lib.DSV_ERR_INVALID_ARG                                                                         # 12 % 8 != 0
    assert L.dsv_cube_permute(FAKE, far, s, *grid, *cube, 2, None) == lib.DSV_ERR_INVALID_ARG          # inverse flag
    assert L.dsv_cube_permute(FAKE, FAKE + 256, s, *grid, *cube, 0, None) == lib.DSV_ERR_INVALID_ARG   # overlap
    assert L.dsv_cube_permute(None, far, s, *grid, *cube, 0, None) == lib.DSV_ERR_INVALID_ARG
    assert L.dsv_cube_permute(FAKE + 8, far, s, *grid, *cube, 0, None) == lib.DSV_ERR_INVALID_ARG      # alignment
    assert L.dsv_cube_permute(FAKE, far, _shape(lib, d=96), *grid, *cube, 0, None) == lib.DSV_ERR_UNSUPPORTED
    assert L.dsv_cube_permute(None, None, _shape(lib, B=0), *grid, *cube, 0, None) == lib.DSV_OK


def test_host_validation_topk_mass(lib):
    L = lib.lib
    s = _shape(lib)                               # nb = 4
    ws = L.dsv_topk_mass_workspace_bytes(s)
    assert ws > L.dsv_topk_workspace_bytes(s)
    cap = 1 * 2 * 4 * 4
    ok = (FAKE, FAKE, FAKE, FAKE)

    def call(tau=0.9, temp=0.1, kmin=1, kmax=4, capacity=cap, wsb=ws, shape=s):
        return L.dsv_topk_mass_blocks(FAKE, shape, tau, temp, kmin, kmax, *ok, capacity, FAKE, wsb, None)
    for bad in (dict(tau=0.0), dict(tau=1.5), dict(tau=float("nan")), dict(temp=0.0), dict(temp=float("inf")),
                dict(kmin=0), dict(kmin=3, kmax=2), dict(kmax=5), dict(capacity=cap - 1), dict(wsb=ws - 1)):
        assert call(**bad) == lib.DSV_ERR_INVALID_ARG, bad
    assert call(shape=_shape(lib, d=96)) == lib.DSV_ERR_UNSUPPORTED
    big = _shape(lib, N=128 * 8193, H=1)
    assert L.dsv_topk_mass_blocks(FAKE, big, 0.9, 0.1, 1, 4, *ok, 1 << 40, FAKE, 1 << 40, None) == \
        lib.DSV_ERR_UNSUPPORTED


def test_host_validation_predict_max(lib):
    L = lib.lib
    s = _shape(lib)
    ws = L.dsv_predict_max_workspace_bytes(s)
    assert ws >= 2 * 1 * 2 * 512 * 48 * 2                  # every token's split row (3r bf16) of Q and of K
    assert L.dsv_predict_max_workspace_bytes(_shape(lib, r=12)) == 0
    ok = (FAKE, FAKE, FAKE, FAKE)
    assert L.dsv_predict_scores_max(*ok, _shape(lib, d=96), FAKE, FAKE, ws, None) == lib.DSV_ERR_UNSUPPORTED
    assert L.dsv_predict_scores_max(*ok, _shape(lib, r=72), FAKE, FAKE, ws, None) == lib.DSV_ERR_UNSUPPORTED
    assert L.dsv_predict_scores_max(*ok, _shape(lib, N=500), FAKE, FAKE, ws, None) == lib.DSV_ERR_INVALID_ARG
    assert L.dsv_predict_scores_max(*ok, s, None, FAKE, ws, None) == lib.DSV_ERR_INVALID_ARG
    assert L.dsv_predict_scores_max(*ok, s, FAKE + 4, FAKE, ws, None) == lib.DSV_ERR_INVALID_ARG
    assert L.dsv_predict_scores_max(*ok, s, FAKE, FAKE + 128, ws, None) == lib.DSV_ERR_INVALID_ARG
    assert L.dsv_predict_scores_max(*ok, s, FAKE, FAKE, ws - 1, None) == lib.DSV_ERR_INVALID_ARG
    assert L.dsv_predict_scores_max(None, None, None, None, _shape(lib, N=0), None, None, 0, None) == lib.DSV_OK


def test_binding_rejects_mismatched_shapes_on_the_host(lib):
    """The binding checks every tensor's shape (and each CSR array's room)
    before the device check and before any call into the library."""
    import torch
    bf = torch.bfloat16
    Q = torch.zeros(1, 2, 256, 64, dtype=bf)             # G = nb = 4 at block 64
    W = torch.zeros(2, 64, 16)
    S = torch.zeros(1, 2, 4, 4)
    i32 = lambda n: torch.zeros(n, dtype=torch.int32)   # noqa: E731
    with pytest.raises(ValueError, match="K has shape"):
        lib.predict_scores(Q, torch.zeros(1, 2, 128, 64, dtype=bf), W, W, 64)
    with pytest.raises(ValueError, match="Wk has shape"):
        lib.predict_scores(Q, Q, W, torch.zeros(2, 64, 8), 64)
    with pytest.raises(ValueError, match="Wq must have 3 dimensions"):
        lib.predict_scores_max(Q, Q, W[0], W, 64)
    with pytest.raises(ValueError, match="out has shape"):
        lib.predict_scores_max(Q, Q, W, W, 64, out=torch.zeros(1, 2, 4, 3))
    with pytest.raises(ValueError, match="scores has shape"):
        lib.topk_blocks(S, [1, 1], 64, 512)
    with pytest.raises(ValueError, match="k_per_head has 1 entries"):
        lib.topk_blocks(S, [1], 64, 256)
    with pytest.raises(ValueError, match="fwd_col holds 15"):
        lib.topk_blocks(S, [2, 2], 64, 256, outs=(i32(9), i32(15), i32(9), i32(16)))
    with pytest.raises(ValueError, match="bwd_ptr holds 8"):
        lib.topk_blocks_noalloc(S, [2, 2], 64, 256, outs=(i32(9), i32(16), i32(8), i32(16)))
    with pytest.raises(ValueError, match="fwd_ptr holds 8"):
        lib.topk_mass_blocks(S, 0.9, 64, 256, outs=(i32(8), i32(32), i32(9), i32(32)))
    with pytest.raises(ValueError, match="V has shape"):
        lib.sparse_attn_fwd(Q, Q, Q[:, :1], i32(9), i32(8), 64)
    with pytest.raises(ValueError, match="fwd_ptr holds 8"):
        lib.sparse_attn_fwd(Q, Q, Q, i32(8), i32(8), 64)
    with pytest.raises(ValueError, match="lse has shape"):
        lib.sparse_attn_fwd(Q, Q, Q, i32(9), i32(8), 64, lse=torch.zeros(1, 2, 255))
    with pytest.raises(ValueError, match="lse has shape"):
        lib.sparse_attn_bwd(Q, Q, Q, Q, Q, torch.zeros(1, 2, 255), i32(9), i32(8), i32(9), i32(8), 64)
    with pytest.raises(ValueError, match="dV has shape"):
        lib.sparse_attn_bwd(Q, Q, Q, Q, Q, torch.zeros(1, 2, 256), i32(9), i32(8), i32(9), i32(8), 64,
                            outs=(Q, Q, Q[..., :32]))
    with pytest.raises(ValueError, match="bwd_ptr holds 4"):
        lib.attn_bwd_dkdv(Q, Q, Q, Q, i32(4), i32(8), 64, outs=(Q, Q), workspace=i32(64))
    with pytest.raises(ValueError, match="dQ has shape"):
        lib.attn_bwd_dq(Q, Q, Q, Q, i32(9), i32(8), 64, out=Q[0], workspace=i32(64))
    with pytest.raises(ValueError, match="dO has shape"):
        lib.attn_bwd_preprocess(Q, Q[:, :, :128], torch.zeros(1, 2, 256), 64, workspace=i32(64))
    with pytest.raises(ValueError, match="out has shape"):
        lib.cube_permute(Q, (4, 8, 8), (1, 8, 8), out=Q[:, :1])
    # consistent shapes reach the device check, still before the library
    with pytest.raises(ValueError, match="CUDA device"):
        lib.predict_scores(Q, Q, W, W, 64)
    with pytest.raises(ValueError, match="CUDA device"):
        lib.sparse_attn_bwd(Q, Q, Q, Q, Q, torch.zeros(1, 2, 256), i32(9), i32(8), i32(9), i32(8), 64)


def test_host_validation_predict_topk(lib):
    L = lib.lib
    s = _shape(lib)
    ws = L.dsv_predict_topk_workspace_bytes(s)
    assert ws >= L.dsv_predict_workspace_bytes(s) + L.dsv_topk_workspace_bytes(s)
    assert L.dsv_predict_topk_workspace_bytes(_shape(lib, r=40)) == 0
    k = (ctypes.c_int32 * 2)(2, 3)
    w4 = (FAKE,) * 4
    outs = (FAKE,) * 4
    assert L.dsv_predict_topk_blocks(*w4, _shape(lib, r=40), k, *outs, None, FAKE, ws, None) == lib.DSV_ERR_UNSUPPORTED
    assert L.dsv_predict_topk_blocks(*w4, _shape(lib, d=96), k, *outs, None, FAKE, ws, None) == lib.DSV_ERR_UNSUPPORTED
    assert L.dsv_predict_topk_blocks(*w4, s, (ctypes.c_int32 * 2)(0, 3), *outs, None, FAKE, ws, None) == \
        lib.DSV_ERR_INVALID_ARG
    assert L.dsv_predict_topk_blocks(*w4, s, (ctypes.c_int32 * 2)(2, 5), *outs, None, FAKE, ws, None) == \
        lib.DSV_ERR_INVALID_ARG
    assert L.dsv_predict_topk_blocks(*w4, s, k, *outs, None, FAKE, ws - 1, None) == lib.DSV_ERR_INVALID_ARG
    assert L.dsv_predict_topk_blocks(*w4, s, k, *outs, FAKE + 4, FAKE, ws, None) == lib.DSV_ERR_INVALID_ARG
    assert L.dsv_predict_topk_blocks(None, FAKE, FAKE, FAKE, s, k, *outs, None, FAKE, ws, None) == \
        lib.DSV_ERR_INVALID_ARG
    assert L.dsv_predict_topk_blocks(*w4, s, k, *outs, None, FAKE + 16, ws, None) == lib.DSV_ERR_INVALID_ARG
    big = _shape(lib, N=128 * 4097, H=1)
    assert L.dsv_predict_topk_blocks(*w4, big, k, *outs, None, FAKE, 1 << 40, None) == lib.DSV_ERR_UNSUPPORTED


def test_noalloc_scratch_holds_every_named_workload(lib):
    """The allocation-free top-k's fixed 64 MiB scratch must hold the top-k
    workspace (selection bitmask, per-segment counts, column totals) of every
    named workload, long518k included (~62 MB)."""
    from dynamic_block_sparse_projection_gb300 import workloads as wl
    for w in wl.WORKLOADS.values():
        need = lib.lib.dsv_topk_workspace_bytes(_shape(lib, B=w.B, H=w.H, N=w.N, d=w.d, block=w.block, r=w.r))
        assert 0 < need <= (64 << 20), (w.name, need)
