"""Thin Python binding of libdsv.so (the C ABI declared in include/dsv.h).

Argument marshalling only: torch tensors supply device memory and the current
CUDA stream; every step of the hot path runs in the library's kernels.  There
is no fallback: if the library has not been built (``__graft_entry__.build()``
or ``python -m dynamic_block_sparse_projection_gb300.build``) importing this
module raises.
"""
from __future__ import annotations

import ctypes
import math
from pathlib import Path
from typing import Optional, Sequence, Tuple

import torch

_LIB_PATH = Path(__file__).resolve().parent / "_build" / "libdsv.so"

DSV_OK, DSV_ERR_INVALID_ARG, DSV_ERR_UNSUPPORTED, DSV_ERR_CUDA, DSV_ERR_BAD_INDEX, DSV_ERR_TIMEOUT, DSV_ERR_INTERNAL = range(7)

# Every symbol the header declares; checked at load time.
EXPORTS = (
    "dsv_predict_workspace_bytes", "dsv_predict_scores",
    "dsv_topk_workspace_bytes", "dsv_topk_blocks",
    "dsv_sparse_attn_fwd",
    "dsv_attn_bwd_workspace_bytes", "dsv_sparse_attn_bwd",
    "dsv_status_string", "dsv_get_device_error", "dsv_clear_device_error",
    "dsv_set_wait_limit_ns", "dsv_version",
    "dsv_topk_blocks_noalloc",
    "dsv_attn_bwd_preprocess", "dsv_attn_bwd_dkdv", "dsv_attn_bwd_dq",
    "dsv_cube_permute", "dsv_topk_mass_workspace_bytes", "dsv_topk_mass_blocks",
    "dsv_predict_max_workspace_bytes", "dsv_predict_scores_max",
    "dsv_selftest_wait_timeout",
    "dsv_predict_topk_workspace_bytes", "dsv_predict_topk_blocks",
    "dsv_dispatch_heads",
)
SELFTEST_WAIT_ID = 0xD5F0


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("N", ctypes.c_int32),
                ("d", ctypes.c_int32), ("block", ctypes.c_int32), ("r", ctypes.c_int32)]


class DsvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def _load() -> ctypes.CDLL:
    if not _LIB_PATH.exists():
        raise ImportError(f"libdsv.so is not built ({_LIB_PATH}); run __graft_entry__.build() first")
    lib = ctypes.CDLL(str(_LIB_PATH))
    missing = [s for s in EXPORTS if not hasattr(lib, s)]
    if missing:
        raise ImportError(f"libdsv.so lacks symbols: {missing}")
    vp, sz, i32, u32p = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.POINTER(ctypes.c_uint32)
    lib.dsv_predict_workspace_bytes.argtypes = [Shape]
    lib.dsv_predict_workspace_bytes.restype = sz
    lib.dsv_predict_scores.argtypes = [vp, vp, vp, vp, Shape, vp, vp, sz, vp]
    lib.dsv_predict_scores.restype = ctypes.c_int
    lib.dsv_predict_max_workspace_bytes.argtypes = [Shape]
    lib.dsv_predict_max_workspace_bytes.restype = sz
    lib.dsv_predict_scores_max.argtypes = [vp, vp, vp, vp, Shape, vp, vp, sz, vp]
    lib.dsv_predict_scores_max.restype = ctypes.c_int
    lib.dsv_topk_workspace_bytes.argtypes = [Shape]
    lib.dsv_topk_workspace_bytes.restype = sz
    lib.dsv_topk_blocks.argtypes = [vp, Shape, ctypes.POINTER(i32), vp, vp, vp, vp, vp, sz, vp]
    lib.dsv_topk_blocks.restype = ctypes.c_int
    lib.dsv_sparse_attn_fwd.argtypes = [vp, vp, vp, Shape, vp, vp, ctypes.c_float, vp, vp, vp]
    lib.dsv_sparse_attn_fwd.restype = ctypes.c_int
    lib.dsv_attn_bwd_workspace_bytes.argtypes = [Shape]
    lib.dsv_attn_bwd_workspace_bytes.restype = sz
    lib.dsv_sparse_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, Shape, vp, vp, vp, vp, ctypes.c_float,
                                        vp, vp, vp, vp, sz, vp]
    lib.dsv_sparse_attn_bwd.restype = ctypes.c_int
    lib.dsv_status_string.argtypes = [ctypes.c_int]
    lib.dsv_status_string.restype = ctypes.c_char_p
    lib.dsv_get_device_error.argtypes = [vp, u32p]
    lib.dsv_get_device_error.restype = ctypes.c_int
    lib.dsv_clear_device_error.argtypes = [vp]
    lib.dsv_clear_device_error.restype = ctypes.c_int
    lib.dsv_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.dsv_set_wait_limit_ns.restype = ctypes.c_int
    lib.dsv_topk_blocks_noalloc.argtypes = [vp, Shape, ctypes.POINTER(i32), vp, vp, vp, vp, vp]
    lib.dsv_topk_blocks_noalloc.restype = ctypes.c_int
    lib.dsv_attn_bwd_preprocess.argtypes = [vp, vp, vp, Shape, vp, sz, vp]
    lib.dsv_attn_bwd_preprocess.restype = ctypes.c_int
    lib.dsv_attn_bwd_dkdv.argtypes = [vp, vp, vp, vp, Shape, vp, vp, ctypes.c_float, vp, vp, vp, sz, vp]
    lib.dsv_attn_bwd_dkdv.restype = ctypes.c_int
    lib.dsv_attn_bwd_dq.argtypes = [vp, vp, vp, vp, Shape, vp, vp, ctypes.c_float, vp, vp, sz, vp]
    lib.dsv_attn_bwd_dq.restype = ctypes.c_int
    lib.dsv_topk_mass_workspace_bytes.argtypes = [Shape]
    lib.dsv_topk_mass_workspace_bytes.restype = sz
    lib.dsv_topk_mass_blocks.argtypes = [vp, Shape, ctypes.c_float, ctypes.c_float, i32, i32, vp, vp, vp, vp, sz, vp,
                                         sz, vp]
    lib.dsv_topk_mass_blocks.restype = ctypes.c_int
    lib.dsv_cube_permute.argtypes = [vp, vp, Shape, i32, i32, i32, i32, i32, i32, i32, vp]
    lib.dsv_cube_permute.restype = ctypes.c_int
    lib.dsv_predict_topk_workspace_bytes.argtypes = [Shape]
    lib.dsv_predict_topk_workspace_bytes.restype = sz
    lib.dsv_predict_topk_blocks.argtypes = [vp, vp, vp, vp, Shape, ctypes.POINTER(i32), vp, vp, vp, vp, vp, vp, sz,
                                            vp]
    lib.dsv_predict_topk_blocks.restype = ctypes.c_int
    f32p = ctypes.POINTER(ctypes.c_float)
    lib.dsv_dispatch_heads.argtypes = [ctypes.POINTER(i32), i32, i32, f32p, f32p, i32, ctypes.POINTER(i32),
                                       ctypes.POINTER(i32)]
    lib.dsv_dispatch_heads.restype = ctypes.c_int
    lib.dsv_selftest_wait_timeout.argtypes = [vp]
    lib.dsv_selftest_wait_timeout.restype = ctypes.c_int
    lib.dsv_version.argtypes = []
    lib.dsv_version.restype = i32
    return lib


lib = _load()


def status_string(status: int) -> str:
    return lib.dsv_status_string(status).decode()


def _check(status: int, what: str) -> None:
    if status != DSV_OK:
        raise DsvError(status, what)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(device: torch.device, stream=None) -> Optional[int]:
    s = torch.cuda.current_stream(device) if stream is None else stream
    return s.cuda_stream


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, device: Optional[torch.device] = None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _dims(t, name: str, n: int) -> Tuple[int, ...]:
    """The shape of t, which must be an n-dimensional tensor."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dim() != n:
        raise ValueError(f"{name} must have {n} dimensions, got shape {tuple(t.shape)}")
    return tuple(int(v) for v in t.shape)


def _shape(t, name: str, shape) -> None:
    """t must have exactly this shape (the library reads and writes whole tensors)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    want = tuple(int(v) for v in shape)
    if tuple(t.shape) != want:
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {want}")


def _room(t, name: str, n: int) -> None:
    """t must hold at least n elements (a CSR array may be longer than its contents)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.numel() < n:
        raise ValueError(f"{name} holds {t.numel()} elements, needs at least {n}")


def _groups(N: int, block: int) -> int:
    return N // block if block > 0 else 0


def _nbytes(t: torch.Tensor) -> int:
    return t.numel() * t.element_size()


def nnz_of(B: int, G: int, k_per_head: Sequence[int]) -> int:
    return B * G * int(sum(int(k) for k in k_per_head))


def _workspace(nbytes: int, device, workspace: Optional[torch.Tensor]) -> torch.Tensor:
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError(f"workspace needs {nbytes} bytes")
        return workspace
    return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)


def predict_workspace_bytes(B: int, H: int, N: int, d: int, block: int, r: int) -> int:
    return lib.dsv_predict_workspace_bytes(Shape(B, H, N, d, block, r))


def topk_workspace_bytes(B: int, H: int, N: int, d: int, block: int) -> int:
    return lib.dsv_topk_workspace_bytes(Shape(B, H, N, d, block, 8))


def attn_bwd_workspace_bytes(B: int, H: int, N: int, d: int, block: int) -> int:
    return lib.dsv_attn_bwd_workspace_bytes(Shape(B, H, N, d, block, 8))


# ---------------------------------------------------------------------------
# The four calls of the hot path
# ---------------------------------------------------------------------------

def predict_scores(Q, K, Wq, Wk, block: int, *, out=None, workspace=None, stream=None) -> torch.Tensor:
    """scores[b,h,g,j] = qbar_g . kbar_j (fp32 [B,H,G,nb]); see dsv_predict_scores."""
    return _predict(lib.dsv_predict_scores, lib.dsv_predict_workspace_bytes, "dsv_predict_scores",
                    Q, K, Wq, Wk, block, out, workspace, stream)


def _predict(fn, ws_fn, what, Q, K, Wq, Wk, block, out, workspace, stream):
    B, H, N, d = _dims(Q, "Q", 4)
    _shape(K, "K", (B, H, N, d))
    r = _dims(Wq, "Wq", 3)[2]
    _shape(Wq, "Wq", (H, d, r))
    _shape(Wk, "Wk", (H, d, r))
    G = _groups(N, block)
    if out is not None:
        _shape(out, "out", (B, H, G, G))
    _need(Q, "Q", torch.bfloat16)
    dev = Q.device
    _need(K, "K", torch.bfloat16, dev)
    _need(Wq, "Wq", torch.float32, dev)
    _need(Wk, "Wk", torch.float32, dev)
    s = Shape(B, H, N, d, block, r)
    if out is None:
        out = torch.empty(B, H, G, G, dtype=torch.float32, device=dev)
    _need(out, "out", torch.float32, dev)
    nbytes = ws_fn(s)
    ws = _workspace(nbytes, dev, workspace)
    with torch.cuda.device(dev):
        _check(fn(_ptr(Q), _ptr(K), _ptr(Wq), _ptr(Wk), s, _ptr(out), _ptr(ws), nbytes, _stream(dev, stream)), what)
    return out


def predict_max_workspace_bytes(B: int, H: int, N: int, d: int, block: int, r: int) -> int:
    return int(lib.dsv_predict_max_workspace_bytes(Shape(B, H, N, d, block, r)))


def predict_scores_max(Q, K, Wq, Wk, block: int, *, out=None, workspace=None, stream=None) -> torch.Tensor:
    """scores[b,h,g,j] = max low-rank logit of tile (g, j) (fp32 [B,H,G,nb]); see dsv_predict_scores_max."""
    return _predict(lib.dsv_predict_scores_max, lib.dsv_predict_max_workspace_bytes, "dsv_predict_scores_max",
                    Q, K, Wq, Wk, block, out, workspace, stream)


def topk_blocks(scores, k_per_head: Sequence[int], block: int, N: int, d: int = 128, *, outs=None,
                workspace=None, stream=None) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor, torch.Tensor]:
    """(fwd_ptr, fwd_col, bwd_ptr, bwd_col) int32 CSR lists; see dsv_topk_blocks."""
    B, H, G, nb = _score_dims(scores, block, N, k_per_head)
    nnz = nnz_of(B, G, k_per_head)
    if outs is not None:
        _csr_room(outs, B * H * G + 1, nnz, B * H * nb + 1, nnz)
    _need(scores, "scores", torch.float32)
    dev = scores.device
    s = Shape(B, H, N, d, block, 8)
    if outs is None:
        outs = (torch.empty(B * H * G + 1, dtype=torch.int32, device=dev),
                torch.empty(max(nnz, 1), dtype=torch.int32, device=dev),
                torch.empty(B * H * nb + 1, dtype=torch.int32, device=dev),
                torch.empty(max(nnz, 1), dtype=torch.int32, device=dev))
    for name, t in zip(("fwd_ptr", "fwd_col", "bwd_ptr", "bwd_col"), outs):
        _need(t, name, torch.int32, dev)
    karr = (ctypes.c_int32 * max(H, 1))(*[int(k) for k in k_per_head])
    nbytes = lib.dsv_topk_workspace_bytes(s)
    ws = _workspace(nbytes, dev, workspace)
    with torch.cuda.device(dev):
        _check(lib.dsv_topk_blocks(_ptr(scores), s, karr, *[_ptr(t) for t in outs], _ptr(ws), nbytes,
                                   _stream(dev, stream)), "dsv_topk_blocks")
    fp, fc, bp, bc = outs
    return fp, fc[:nnz], bp, bc[:nnz]


def predict_topk_workspace_bytes(B: int, H: int, N: int, d: int, block: int, r: int) -> int:
    return int(lib.dsv_predict_topk_workspace_bytes(Shape(B, H, N, d, block, r)))


def predict_topk_blocks(Q, K, Wq, Wk, k_per_head: Sequence[int], block: int, *, outs=None, scores=None,
                        workspace=None, stream=None) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor, torch.Tensor]:
    """(fwd_ptr, fwd_col, bwd_ptr, bwd_col) int32 CSR lists of the fused
    predictor + top-k (the score matrix stays on chip); see
    dsv_predict_topk_blocks.  `scores`, if given (fp32 [B, H, G, G]),
    receives the scores the selection used."""
    B, H, N, d = _dims(Q, "Q", 4)
    _shape(K, "K", (B, H, N, d))
    r = _dims(Wq, "Wq", 3)[2]
    _shape(Wq, "Wq", (H, d, r))
    _shape(Wk, "Wk", (H, d, r))
    if len(k_per_head) != H:
        raise ValueError(f"k_per_head has {len(k_per_head)} entries, expected one per head ({H})")
    G = _groups(N, block)
    nnz = nnz_of(B, G, k_per_head)
    if outs is not None:
        _csr_room(outs, B * H * G + 1, nnz, B * H * G + 1, nnz)
    if scores is not None:
        _shape(scores, "scores", (B, H, G, G))
    _need(Q, "Q", torch.bfloat16)
    dev = Q.device
    _need(K, "K", torch.bfloat16, dev)
    _need(Wq, "Wq", torch.float32, dev)
    _need(Wk, "Wk", torch.float32, dev)
    if scores is not None:
        _need(scores, "scores", torch.float32, dev)
    if outs is None:
        outs = (torch.empty(B * H * G + 1, dtype=torch.int32, device=dev),
                torch.empty(max(nnz, 1), dtype=torch.int32, device=dev),
                torch.empty(B * H * G + 1, dtype=torch.int32, device=dev),
                torch.empty(max(nnz, 1), dtype=torch.int32, device=dev))
    for name, t in zip(("fwd_ptr", "fwd_col", "bwd_ptr", "bwd_col"), outs):
        _need(t, name, torch.int32, dev)
    s = Shape(B, H, N, d, block, r)
    karr = (ctypes.c_int32 * max(H, 1))(*[int(k) for k in k_per_head])
    nbytes = lib.dsv_predict_topk_workspace_bytes(s)
    ws = _workspace(nbytes, dev, workspace)
    with torch.cuda.device(dev):
        _check(lib.dsv_predict_topk_blocks(_ptr(Q), _ptr(K), _ptr(Wq), _ptr(Wk), s, karr, *[_ptr(t) for t in outs],
                                           _ptr(scores), _ptr(ws), nbytes, _stream(dev, stream)),
               "dsv_predict_topk_blocks")
    fp, fc, bp, bc = outs
    return fp, fc[:nnz], bp, bc[:nnz]


def _score_dims(scores, block: int, N: int, k_per_head=None) -> Tuple[int, int, int, int]:
    """[B, H, G, nb] of a score matrix, which must be square with G = N / block."""
    B, H, G, nb = _dims(scores, "scores", 4)
    if G != nb or G != _groups(N, block):
        raise ValueError(f"scores has shape {(B, H, G, nb)}, expected [B, H, N/block, N/block] "
                         f"with N = {N}, block = {block}")
    if k_per_head is not None and len(k_per_head) != H:
        raise ValueError(f"k_per_head has {len(k_per_head)} entries, expected one per head ({H})")
    return B, H, G, nb


def _csr_room(outs, n_fptr: int, n_fcol: int, n_bptr: int, n_bcol: int) -> None:
    if len(outs) != 4:
        raise ValueError("outs must be (fwd_ptr, fwd_col, bwd_ptr, bwd_col)")
    for name, t, n in zip(("fwd_ptr", "fwd_col", "bwd_ptr", "bwd_col"), outs, (n_fptr, n_fcol, n_bptr, n_bcol)):
        _room(t, name, n)


def topk_mass_workspace_bytes(B: int, H: int, N: int, d: int, block: int) -> int:
    return lib.dsv_topk_mass_workspace_bytes(Shape(B, H, N, d, block, 8))


def topk_mass_blocks(scores, tau: float, block: int, N: int, d: int = 128, *, temperature: float = 0.0,
                     kmin: int = 1, kmax: int = 0, outs=None, workspace=None, stream=None, trim: bool = True):
    """(fwd_ptr, fwd_col, bwd_ptr, bwd_col) int32 CSR lists of the
    mass-threshold selection; see dsv_topk_mass_blocks.  temperature <= 0
    selects 1/sqrt(d), kmax <= 0 selects nb.  With trim the column arrays are
    returned cut to nnz = fwd_ptr[-1], which this reads back from the device
    (a synchronisation); without it they are returned whole."""
    B, H, G, nb = _score_dims(scores, block, N)
    if outs is not None:
        _csr_room(outs, B * H * G + 1, 0, B * H * nb + 1, 0)     # the columns' capacity goes to the library
    _need(scores, "scores", torch.float32)
    dev = scores.device
    s = Shape(B, H, N, d, block, 8)
    temperature = float(temperature) if temperature > 0 else 1.0 / math.sqrt(d)
    kmax = int(kmax) if kmax > 0 else nb
    cap = B * H * G * kmax
    if outs is None:
        outs = (torch.empty(B * H * G + 1, dtype=torch.int32, device=dev),
                torch.empty(max(cap, 1), dtype=torch.int32, device=dev),
                torch.empty(B * H * nb + 1, dtype=torch.int32, device=dev),
                torch.empty(max(cap, 1), dtype=torch.int32, device=dev))
    for name, t in zip(("fwd_ptr", "fwd_col", "bwd_ptr", "bwd_col"), outs):
        _need(t, name, torch.int32, dev)
    cap = min(outs[1].numel(), outs[3].numel())
    nbytes = lib.dsv_topk_mass_workspace_bytes(s)
    ws = _workspace(nbytes, dev, workspace)
    with torch.cuda.device(dev):
        _check(lib.dsv_topk_mass_blocks(_ptr(scores), s, float(tau), temperature, int(kmin), kmax,
                                        *[_ptr(t) for t in outs], cap, _ptr(ws), nbytes, _stream(dev, stream)),
               "dsv_topk_mass_blocks")
    fp, fc, bp, bc = outs
    if not trim:
        return fp, fc, bp, bc
    nnz = int(fp[-1].item()) if B * H * G > 0 else 0
    return fp, fc[:nnz], bp, bc[:nnz]


def topk_blocks_noalloc(scores, k_per_head: Sequence[int], block: int, N: int, d: int = 128, *, outs,
                        stream=None) -> None:
    """dsv_topk_blocks_noalloc into caller-provided `outs`; it allocates nothing.

    For callers that cannot allocate device memory: the library's fixed
    device scratch replaces the workspace.  Calls share that scratch, so do
    not let two of them overlap on the GPU.
    """
    B, H, G, nb = _score_dims(scores, block, N, k_per_head)
    nnz = nnz_of(B, G, k_per_head)
    _csr_room(outs, B * H * G + 1, nnz, B * H * nb + 1, nnz)
    _need(scores, "scores", torch.float32)
    dev = scores.device
    for name, t in zip(("fwd_ptr", "fwd_col", "bwd_ptr", "bwd_col"), outs):
        _need(t, name, torch.int32, dev)
    karr = (ctypes.c_int32 * max(H, 1))(*[int(k) for k in k_per_head])
    with torch.cuda.device(dev):
        _check(lib.dsv_topk_blocks_noalloc(_ptr(scores), Shape(B, H, N, d, block, 8), karr,
                                           *[_ptr(t) for t in outs], _stream(dev, stream)), "dsv_topk_blocks_noalloc")


def sparse_attn_fwd(Q, K, V, fwd_ptr, fwd_col, block: int, softmax_scale: float = 0.0, *, out=None, lse=None,
                    stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """(O bf16 [B,H,N,d], lse fp32 [B,H,N]); see dsv_sparse_attn_fwd."""
    B, H, N, d = _dims(Q, "Q", 4)
    for name, t in (("K", K), ("V", V)) + ((("out", out),) if out is not None else ()):
        _shape(t, name, (B, H, N, d))
    if lse is not None:
        _shape(lse, "lse", (B, H, N))
    _room(fwd_ptr, "fwd_ptr", B * H * _groups(N, block) + 1)
    _need(Q, "Q", torch.bfloat16)
    dev = Q.device
    for name, t in (("K", K), ("V", V)):
        _need(t, name, torch.bfloat16, dev)
    for name, t in (("fwd_ptr", fwd_ptr), ("fwd_col", fwd_col)):
        _need(t, name, torch.int32, dev)
    B, H, N, d = Q.shape
    s = Shape(B, H, N, d, block, 8)
    if out is None:
        out = torch.empty_like(Q)
    if lse is None:
        lse = torch.empty(B, H, N, dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, dev)
    _need(lse, "lse", torch.float32, dev)
    with torch.cuda.device(dev):
        _check(lib.dsv_sparse_attn_fwd(_ptr(Q), _ptr(K), _ptr(V), s, _ptr(fwd_ptr), _ptr(fwd_col),
                                       float(softmax_scale), _ptr(out), _ptr(lse), _stream(dev, stream)),
               "dsv_sparse_attn_fwd")
    return out, lse


def sparse_attn_bwd(Q, K, V, O, dO, lse, fwd_ptr, fwd_col, bwd_ptr, bwd_col, block: int,
                    softmax_scale: float = 0.0, *, outs=None, workspace=None, stream=None):
    """(dQ, dK, dV) bf16 [B,H,N,d]; see dsv_sparse_attn_bwd."""
    B, H, N, d = _dims(Q, "Q", 4)
    for name, t in (("K", K), ("V", V), ("O", O), ("dO", dO)):
        _shape(t, name, (B, H, N, d))
    if outs is not None:
        if len(outs) != 3:
            raise ValueError("outs must be (dQ, dK, dV)")
        for name, t in zip(("dQ", "dK", "dV"), outs):
            _shape(t, name, (B, H, N, d))
    _shape(lse, "lse", (B, H, N))
    rows = B * H * _groups(N, block) + 1
    _room(fwd_ptr, "fwd_ptr", rows)
    _room(bwd_ptr, "bwd_ptr", rows)
    _need(Q, "Q", torch.bfloat16)
    dev = Q.device
    for name, t in (("K", K), ("V", V), ("O", O), ("dO", dO)):
        _need(t, name, torch.bfloat16, dev)
    _need(lse, "lse", torch.float32, dev)
    for name, t in (("fwd_ptr", fwd_ptr), ("fwd_col", fwd_col), ("bwd_ptr", bwd_ptr), ("bwd_col", bwd_col)):
        _need(t, name, torch.int32, dev)
    B, H, N, d = Q.shape
    s = Shape(B, H, N, d, block, 8)
    if outs is None:
        outs = (torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V))
    for name, t in zip(("dQ", "dK", "dV"), outs):
        _need(t, name, torch.bfloat16, dev)
    nbytes = lib.dsv_attn_bwd_workspace_bytes(s)
    ws = _workspace(nbytes, dev, workspace)
    with torch.cuda.device(dev):
        _check(lib.dsv_sparse_attn_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(lse), s,
                                       _ptr(fwd_ptr), _ptr(fwd_col), _ptr(bwd_ptr), _ptr(bwd_col),
                                       float(softmax_scale), *[_ptr(t) for t in outs], _ptr(ws), nbytes,
                                       _stream(dev, stream)), "dsv_sparse_attn_bwd")
    return outs


def cube_permute(x, grid, cube, *, inverse: bool = False, out=None, stream=None) -> torch.Tensor:
    """x bf16 [B,H,N,d] between raster and cube token order; see dsv_cube_permute.

    grid = (T, Hl, Wl) with N = T*Hl*Wl; cube = (ct, cy, cx), whose volume is
    the group / block size of the hot path."""
    _dims(x, "x", 4)
    if out is not None:
        _shape(out, "out", x.shape)
    _need(x, "x", torch.bfloat16)
    dev = x.device
    B, H, N, d = x.shape
    T, Hl, Wl = (int(v) for v in grid)
    ct, cy, cx = (int(v) for v in cube)
    if out is None:
        out = torch.empty_like(x)
    _need(out, "out", torch.bfloat16, dev)
    s = Shape(B, H, N, d, ct * cy * cx, 8)
    with torch.cuda.device(dev):
        _check(lib.dsv_cube_permute(_ptr(x), _ptr(out), s, T, Hl, Wl, ct, cy, cx, 1 if inverse else 0,
                                    _stream(dev, stream)), "dsv_cube_permute")
    return out


def attn_bwd_preprocess(O, dO, lse, block: int, *, workspace, stream=None) -> None:
    """D and lse * log2(e) into `workspace`; see dsv_attn_bwd_preprocess."""
    B, H, N, d = _dims(O, "O", 4)
    _shape(dO, "dO", (B, H, N, d))
    _shape(lse, "lse", (B, H, N))
    _need(O, "O", torch.bfloat16)
    dev = O.device
    _need(dO, "dO", torch.bfloat16, dev)
    _need(lse, "lse", torch.float32, dev)
    _need(workspace, "workspace", workspace.dtype, dev)
    s = Shape(B, H, N, d, block, 8)
    with torch.cuda.device(dev):
        _check(lib.dsv_attn_bwd_preprocess(_ptr(O), _ptr(dO), _ptr(lse), s, _ptr(workspace), _nbytes(workspace),
                                           _stream(dev, stream)), "dsv_attn_bwd_preprocess")


def attn_bwd_dkdv(Q, K, V, dO, bwd_ptr, bwd_col, block: int, softmax_scale: float = 0.0, *, outs, workspace,
                  stream=None) -> None:
    """dK, dV into outs = (dK, dV) after attn_bwd_preprocess; see dsv_attn_bwd_dkdv."""
    B, H, N, d = _dims(Q, "Q", 4)
    if len(outs) != 2:
        raise ValueError("outs must be (dK, dV)")
    for name, t in (("K", K), ("V", V), ("dO", dO), ("dK", outs[0]), ("dV", outs[1])):
        _shape(t, name, (B, H, N, d))
    _room(bwd_ptr, "bwd_ptr", B * H * _groups(N, block) + 1)
    _need(Q, "Q", torch.bfloat16)
    dev = Q.device
    for name, t in (("K", K), ("V", V), ("dO", dO), ("dK", outs[0]), ("dV", outs[1])):
        _need(t, name, torch.bfloat16, dev)
    for name, t in (("bwd_ptr", bwd_ptr), ("bwd_col", bwd_col)):
        _need(t, name, torch.int32, dev)
    B, H, N, d = Q.shape
    s = Shape(B, H, N, d, block, 8)
    _need(workspace, "workspace", workspace.dtype, dev)
    with torch.cuda.device(dev):
        _check(lib.dsv_attn_bwd_dkdv(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), s, _ptr(bwd_ptr), _ptr(bwd_col),
                                     float(softmax_scale), _ptr(outs[0]), _ptr(outs[1]), _ptr(workspace),
                                     _nbytes(workspace), _stream(dev, stream)), "dsv_attn_bwd_dkdv")


def attn_bwd_dq(Q, K, V, dO, fwd_ptr, fwd_col, block: int, softmax_scale: float = 0.0, *, out, workspace,
                stream=None) -> None:
    """dQ into `out` after attn_bwd_preprocess; see dsv_attn_bwd_dq."""
    B, H, N, d = _dims(Q, "Q", 4)
    for name, t in (("K", K), ("V", V), ("dO", dO), ("dQ", out)):
        _shape(t, name, (B, H, N, d))
    _room(fwd_ptr, "fwd_ptr", B * H * _groups(N, block) + 1)
    _need(Q, "Q", torch.bfloat16)
    dev = Q.device
    for name, t in (("K", K), ("V", V), ("dO", dO), ("dQ", out)):
        _need(t, name, torch.bfloat16, dev)
    for name, t in (("fwd_ptr", fwd_ptr), ("fwd_col", fwd_col)):
        _need(t, name, torch.int32, dev)
    B, H, N, d = Q.shape
    s = Shape(B, H, N, d, block, 8)
    _need(workspace, "workspace", workspace.dtype, dev)
    with torch.cuda.device(dev):
        _check(lib.dsv_attn_bwd_dq(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), s, _ptr(fwd_ptr), _ptr(fwd_col),
                                   float(softmax_scale), _ptr(out), _ptr(workspace), _nbytes(workspace),
                                   _stream(dev, stream)), "dsv_attn_bwd_dq")


# ---------------------------------------------------------------------------
# Device-side error word
# ---------------------------------------------------------------------------

def device_error(stream=None, device=None) -> Tuple[int, int]:
    """(status, info) recorded by the kernels on the current device; synchronises."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    info = ctypes.c_uint32(0)
    st = lib.dsv_get_device_error(_stream(dev, stream), ctypes.byref(info))
    return st, info.value


def clear_device_error(stream=None, device=None) -> None:
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    _check(lib.dsv_clear_device_error(_stream(dev, stream)), "dsv_clear_device_error")


def set_wait_limit_ns(limit_ns: int) -> None:
    _check(lib.dsv_set_wait_limit_ns(int(limit_ns)), "dsv_set_wait_limit_ns")



def selftest_wait_timeout(stream=None, device=None) -> None:
    """Enqueue the library's failure-detection self-test: a kernel whose only
    wait can never be satisfied runs out of its time limit (set_wait_limit_ns)
    and records DSV_ERR_TIMEOUT; read it with device_error()."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    _check(lib.dsv_selftest_wait_timeout(_stream(dev, stream)), "dsv_selftest_wait_timeout")


def dispatch_heads(k_per_head: Sequence[int], nb: int, rho: Sequence[float], ratio: Sequence[float]):
    """The OP dispatcher (host-only): per head, dense (k = nb) when the profile's
    sparse/dense time ratio at the head's kept fraction is >= 1, else sparse.
    Returns (k_out, dense) as lists; see dsv_dispatch_heads."""
    H, n = len(k_per_head), len(rho)
    if len(ratio) != n:
        raise ValueError("rho and ratio must have the same length")
    karr = (ctypes.c_int32 * max(H, 1))(*[int(k) for k in k_per_head])
    rarr = (ctypes.c_float * max(n, 1))(*[float(v) for v in rho])
    qarr = (ctypes.c_float * max(n, 1))(*[float(v) for v in ratio])
    kout = (ctypes.c_int32 * max(H, 1))()
    dout = (ctypes.c_int32 * max(H, 1))()
    _check(lib.dsv_dispatch_heads(karr, H, int(nb), rarr, qarr, n, kout, dout), "dsv_dispatch_heads")
    return [int(kout[h]) for h in range(H)], [bool(dout[h]) for h in range(H)]
