"""The seeded workload generator: shapes, k rounding, determinism (CPU only)."""
import math

import torch

from dynamic_block_sparse_projection_gb300 import workloads as wl


def test_k_per_head_rounding():
    assert wl.head_params(wl.WORKLOADS["tiny"])[0] == [2, 2]
    assert wl.head_params(wl.WORKLOADS["latent16k"])[0] == [13] * 24
    assert wl.head_params(wl.WORKLOADS["latent123k_global"])[0] == [96] * 24
    assert wl.head_params(wl.WORKLOADS["long518k"])[0] == [203] * 24
    ks, sig, _ = wl.head_params(wl.WORKLOADS["stress61k"])
    assert len(ks) == 16 and all(math.ceil(0.05 * 480) <= k <= math.ceil(0.30 * 480) for k in ks)
    assert all(0.5 <= s <= 3.0 for s in sig)
    _, _, glob = wl.head_params(wl.WORKLOADS["latent123k_global"])
    assert all(len(set(g)) == 4 and all(0 <= j < 960 for j in g) for g in glob)


def test_posemb_bands():
    pe = wl.posemb_3d(4, 8, 8, 64).double()
    c = 2 * (64 // 6)
    assert torch.all(pe[:, 3 * c:] == 0)
    for a in range(3):
        band = pe[:, a * c:(a + 1) * c]
        assert torch.allclose(band[:, 0::2] ** 2 + band[:, 1::2] ** 2, torch.ones(256, c // 2, dtype=torch.float64), atol=1e-6)
    # token n = (t*8 + y)*8 + x: the t band of tokens 0 and 64 differs, x band of 0 and 1 differs
    assert not torch.allclose(pe[0, :c], pe[64, :c]) and torch.allclose(pe[0, c:2 * c], pe[64, c:2 * c])


def test_tiny_inputs_deterministic_and_shaped():
    w = wl.WORKLOADS["tiny"]
    a = wl.make_inputs(w)
    b = wl.make_inputs(w)
    assert a.Q.shape == (1, 2, 256, 64) and a.Q.dtype == torch.bfloat16
    assert a.Wq.shape == (2, 64, 16) and a.Wq.dtype == torch.float32
    for x, y in ((a.Q, b.Q), (a.K, b.K), (a.V, b.V), (a.dO, b.dO), (a.Wq, b.Wq)):
        assert torch.equal(x, y)
    sub = wl.make_inputs(w, heads=[1])
    assert torch.equal(sub.Q[0, 0], a.Q[0, 1]) and torch.equal(sub.Wk[0], a.Wk[1])
