"""Seeded synthetic video-latent workloads for the DSV sparse-attention hot path.

This module only draws inputs.  It holds none of the method's arithmetic (no
pooling, no scoring, no selection, no attention), so both the CUDA path and the
fp64 oracle can be fed from it without sharing any computation.

Workloads stand in for the latent tokens of a video Diffusion Transformer (the
DSV pages, "Technische samenvatting" section 1 and 4: latents of 100k-520k
tokens).  No dataset or trained weights are used: Q, K and V are N(0,1) noise
plus a 3D sinusoidal positional embedding, which gives the attention the
spatio-temporal locality the pages describe (adjacent tokens in 3D space share
critical KV, section 2B), and the low-rank predictor weights are random
N(0, 1/d) matrices (the pages' stage-1 predictor training is not reproduced).

Token order is raster order over the latent grid: n = (t * Hl + y) * Wl + x.
Groups (queries) and blocks (keys) are `block` consecutive tokens.

Seeds: each tensor has its own torch.Generator seeded with 1000 * seed + id
(Q 1, K 2, V 3, dO 4, Wq 5, Wk 6, per-head parameters 7, samples 8).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Tuple

import torch

GEN_Q, GEN_K, GEN_V, GEN_DO, GEN_WQ, GEN_WK, GEN_HEAD, GEN_SAMPLE = 1, 2, 3, 4, 5, 6, 7, 8


@dataclass(frozen=True)
class Workload:
    """Shape and structure of one synthetic workload.

    keep_pct: keep ceil(keep_pct/100 * nb) blocks per group (every head), or
    keep_count: a fixed k per group, or keep_range: per-head keep ratio drawn
    U[lo, hi] from the per-head generator.
    """
    name: str
    B: int
    H: int
    d: int
    T: int
    Hl: int
    Wl: int
    block: int
    r: int
    seed: int
    keep_count: Optional[int] = None
    keep_pct: Optional[int] = None
    keep_range: Optional[Tuple[float, float]] = None
    sigma: float = 2.0
    sigma_range: Optional[Tuple[float, float]] = None
    n_global: int = 0
    global_gain: float = 1.0
    description: str = ""

    @property
    def N(self) -> int:
        return self.T * self.Hl * self.Wl

    @property
    def nb(self) -> int:
        return self.N // self.block


WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny", B=1, H=2, d=64, T=4, Hl=8, Wl=8, block=64, r=16, seed=0,
                 keep_count=2,
                 description="B1 H2 d64, latent 4x8x8=256 tokens, block 64 (4 KV blocks), r16, top-2"),
        Workload("latent16k", B=1, H=24, d=128, T=16, Hl=32, Wl=32, block=128, r=16, seed=1,
                 keep_pct=10,
                 description="B1 H24 d128, latent 16x32x32=16384 tokens, block 128 (128 KV blocks), r16, top 10% (13)"),
        Workload("latent123k_global", B=1, H=24, d=128, T=32, Hl=48, Wl=80, block=128, r=32, seed=2,
                 keep_pct=10, n_global=4, global_gain=3.0,
                 description="B1 H24 d128, latent 32x48x80=122880 tokens, block 128 (960 KV blocks), r32, "
                             "top 10% (96), 4 global key blocks per head amplified 3x"),
        Workload("stress61k", B=2, H=16, d=128, T=24, Hl=40, Wl=64, block=128, r=32, seed=3,
                 keep_range=(0.05, 0.30), sigma_range=(0.5, 3.0),
                 description="B2 H16 d128, latent 24x40x64=61440 tokens, block 128 (480 KV blocks), r32, "
                             "per-head keep U[5%,30%], per-head pos-emb scale U[0.5,3]"),
        Workload("long518k", B=1, H=24, d=128, T=64, Hl=90, Wl=90, block=128, r=32, seed=4,
                 keep_pct=5,
                 description="B1 H24 d128, latent 64x90x90=518400 tokens, block 128 (4050 KV blocks), r32, "
                             "top 5% (203)"),
    ]
}


def _gen(seed: int, gid: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(1000 * seed + gid)
    return g


def head_params(w: Workload) -> Tuple[List[int], List[float], List[List[int]]]:
    """Per-head k, pos-emb scale and 'global' key blocks, drawn on the CPU.

    k rounding: k = ceil(p * nb) clamped to [1, nb].
    """
    g = _gen(w.seed, GEN_HEAD, "cpu")
    nb = w.nb
    if w.keep_count is not None:
        ks = [w.keep_count] * w.H
    elif w.keep_pct is not None:
        ks = [(w.keep_pct * nb + 99) // 100] * w.H
    else:
        lo, hi = w.keep_range
        rho = torch.rand(w.H, generator=g, dtype=torch.float64) * (hi - lo) + lo
        ks = [int(math.ceil(float(p) * nb)) for p in rho]
    ks = [max(1, min(nb, k)) for k in ks]
    if w.sigma_range is not None:
        lo, hi = w.sigma_range
        sig = (torch.rand(w.H, generator=g, dtype=torch.float64) * (hi - lo) + lo).tolist()
    else:
        sig = [w.sigma] * w.H
    globals_: List[List[int]] = []
    for _ in range(w.H):
        if w.n_global:
            globals_.append(sorted(torch.randperm(nb, generator=g)[: w.n_global].tolist()))
        else:
            globals_.append([])
    return ks, sig, globals_


def posemb_3d(T: int, Hl: int, Wl: int, d: int, device="cpu") -> torch.Tensor:
    """3D sinusoidal positional embedding [T*Hl*Wl, d] in fp32.

    d is split into three axis bands (t, y, x) of c = 2*floor(d/6) channels;
    channels past 3c are zero.  In a band with integer coordinate p, channel
    pair (2i, 2i+1) holds (sin(p*w_i), cos(p*w_i)), w_i = 10000^(-2i/c).
    """
    c = 2 * (d // 6)
    half = c // 2
    i = torch.arange(half, dtype=torch.float64, device=device)
    omega = torch.pow(torch.tensor(10000.0, dtype=torch.float64, device=device), -2.0 * i / c)
    n = torch.arange(T * Hl * Wl, device=device)
    coords = [n // (Hl * Wl), (n // Wl) % Hl, n % Wl]
    pe = torch.zeros(T * Hl * Wl, d, dtype=torch.float64, device=device)
    for a, p in enumerate(coords):
        ang = p.to(torch.float64)[:, None] * omega[None, :]
        pe[:, a * c: a * c + c: 2] = torch.sin(ang)
        pe[:, a * c + 1: a * c + c: 2] = torch.cos(ang)
    return pe.to(torch.float32)


@dataclass
class Inputs:
    w: Workload
    Q: torch.Tensor   # [B,H,N,d] bf16
    K: torch.Tensor
    V: torch.Tensor
    dO: Optional[torch.Tensor]
    Wq: torch.Tensor  # [H,d,r] fp32
    Wk: torch.Tensor
    k_per_head: List[int]
    sigma: List[float]
    global_blocks: List[List[int]] = field(default_factory=list)


def make_inputs(w: Workload, device="cpu", with_dO: bool = True, heads: Optional[List[int]] = None) -> Inputs:
    """Draw one workload's tensors on `device` (bf16 activations, fp32 weights).

    Every head is drawn in turn from the same per-tensor generator, so the
    values do not depend on how many heads are kept: `heads` selects a subset
    after drawing (used to cut host memory when only a few heads are needed).
    """
    ks, sig, glob = head_params(w)
    B, H, N, d, r = w.B, w.H, w.N, w.d, w.r
    pe = posemb_3d(w.T, w.Hl, w.Wl, d, device=device)
    keep = list(range(H)) if heads is None else list(heads)
    gens = {gid: _gen(w.seed, gid, device) for gid in (GEN_Q, GEN_K, GEN_V, GEN_DO)}
    out = {}
    for name, gid in (("Q", GEN_Q), ("K", GEN_K), ("V", GEN_V), ("dO", GEN_DO)):
        if name == "dO" and not with_dO:
            continue
        t = torch.empty(B, len(keep), N, d, dtype=torch.bfloat16, device=device)
        for b in range(B):
            for h in range(H):
                x = torch.randn(N, d, generator=gens[gid], device=device, dtype=torch.float32)
                if h not in keep:
                    continue
                if name != "dO":
                    x = x + sig[h] * pe
                if name == "K" and glob[h]:
                    for j in glob[h]:
                        x[j * w.block:(j + 1) * w.block] *= w.global_gain
                t[b, keep.index(h)] = x.to(torch.bfloat16)
        out[name] = t
    gw = {gid: _gen(w.seed, gid, device) for gid in (GEN_WQ, GEN_WK)}
    Wq = (torch.randn(H, d, r, generator=gw[GEN_WQ], device=device, dtype=torch.float32) / math.sqrt(d))[keep].contiguous()
    Wk = (torch.randn(H, d, r, generator=gw[GEN_WK], device=device, dtype=torch.float32) / math.sqrt(d))[keep].contiguous()
    return Inputs(w=w, Q=out["Q"], K=out["K"], V=out["V"], dO=out.get("dO"), Wq=Wq, Wk=Wk,
                  k_per_head=[ks[h] for h in keep], sigma=[sig[h] for h in keep],
                  global_blocks=[glob[h] for h in keep])


def scaled(w: Workload, *, name: Optional[str] = None, **changes) -> Workload:
    """A copy of `w` with some fields changed (smaller parity-test variants)."""
    fields = dict(w.__dict__)
    fields.update(changes)
    fields["name"] = name or (w.name + "_small")
    return Workload(**fields)


def sample_indices(n: int, count: int, seed: int, gid: int = GEN_SAMPLE) -> List[int]:
    """`count` distinct seeded indices in [0, n), ascending."""
    g = _gen(seed, gid, "cpu")
    count = min(count, n)
    return sorted(torch.randperm(n, generator=g)[:count].tolist())
