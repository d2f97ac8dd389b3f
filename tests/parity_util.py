"""Shared helpers of the GPU parity tests (comparison rules and small workloads)."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from dynamic_block_sparse_projection_gb300 import workloads as wl

# Tolerances of the hot path.
SCORE_REL = 1e-4          # |dS| <= 1e-4 * max(|S_ref|, rms of the S_ref row)
O_REL_L2, O_MAX_ABS = 1e-2, 2e-2
GRAD_REL_L2 = 2e-2
LSE_MAX_ABS = 2e-2        # reported alongside O


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def rel_l2(x, y) -> float:
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    den = np.linalg.norm(y.ravel())
    return float(np.linalg.norm((x - y).ravel()) / (den if den > 0 else 1.0))


def bf16_half_ulp(ref) -> np.ndarray:
    """Half the spacing of the bf16 grid at each reference value (|x| >= 2^-126)."""
    r = np.abs(np.asarray(ref, np.float64)).astype(np.float32)
    return np.spacing(r).astype(np.float64) * 2.0 ** 15


def max_abs_beyond_rounding(gpu, ref) -> float:
    """max |gpu - ref| less the half-ulp that storing ref in bf16 alone can cost.

    O is a bf16 output: above |O| = 4 half a bf16 ulp is already 0.0156, and
    above 8 it exceeds the 2e-2 bar by itself, so the max-abs bar is applied
    to the error beyond the output format's own rounding.
    """
    g = np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    return float(np.max(np.abs(g - r) - bf16_half_ulp(r))) if g.size else 0.0


def score_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    """max |gpu - ref| / max(|ref|, rms(ref row)) over all entries."""
    rms = np.sqrt(np.mean(ref ** 2, axis=-1, keepdims=True))
    den = np.maximum(np.abs(ref), rms)
    den = np.where(den > 0, den, 1.0)
    return float(np.max(np.abs(gpu - ref) / den)) if gpu.size else 0.0


# Reduced variants of the workloads: same structure, sizes the oracle finishes
# in seconds, several tiles per (b, h) and ragged bitmask words.
SMALL = {
    "latent16k_small": wl.scaled(wl.WORKLOADS["latent16k"], name="latent16k_small", H=2, T=4),
    "global_small": wl.scaled(wl.WORKLOADS["latent123k_global"], name="global_small", H=2, T=37, Hl=8, Wl=16),
    "stress_small": wl.scaled(wl.WORKLOADS["stress61k"], name="stress_small", H=3, T=12, Hl=10, Wl=16),
    "long_small": wl.scaled(wl.WORKLOADS["long518k"], name="long_small", H=1, T=40, Hl=8, Wl=16),
}


def oracle_lists(S64: np.ndarray, ks, G: int):
    B, H = S64.shape[:2]
    fp, fc = oracle.topk_lists(S64, ks)
    bp, bc = oracle.transpose_lists(fp, fc, B, H, G, G)
    return fp, fc, bp, bc


def csr_to_device(arrs, device):
    return [torch.as_tensor(np.asarray(a, dtype=np.int32), device=device) for a in arrs]


def random_lists(rng, B, H, G, ks):
    ptr = [0]
    col = []
    for _b in range(B):
        for h in range(H):
            for _g in range(G):
                sel = np.sort(rng.choice(G, size=ks[h], replace=False))
                col.extend(sel.tolist())
                ptr.append(ptr[-1] + ks[h])
    fp, fc = np.array(ptr), np.array(col)
    bp, bc = oracle.transpose_lists(fp, fc, B, H, G, G)
    return fp, fc, bp, bc


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)
