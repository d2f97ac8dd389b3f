"""The allocation-free top-k entry point (needs a GB300).

dsv_topk_blocks_noalloc serves callers that cannot allocate device memory:
code running while another thread captures a CUDA graph, plug-ins whose host
framework owns the device heap, loops where an allocation may block.  It
draws its scratch from a fixed array inside libdsv instead of a workspace.

Checked through the C ABI: two calls in a row give exactly the lists of the
allocating dsv_topk_blocks (index work: bit-exact), for two different shapes
so that the shared scratch's leftover contents cannot leak into a result; and
a problem larger than the fixed scratch is refused before any launch.  This
file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from dynamic_block_sparse_projection_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dynamic_block_sparse_projection_gb300 import binding
    return binding


def _raw_noalloc(dsv, S, ks, w, outs):
    B, H, G, _ = S.shape
    karr = (ctypes.c_int32 * H)(*ks)
    stream = torch.cuda.current_stream().cuda_stream
    return dsv.lib.dsv_topk_blocks_noalloc(S.data_ptr(), dsv.Shape(B, H, w.N, w.d, w.block, 8), karr,
                                           *[t.data_ptr() for t in outs], stream)


@pytest.mark.parametrize("name", ["latent16k", "stress61k"])
def test_noalloc_matches_allocating_topk_twice(dsv, name):
    w = wl.WORKLOADS[name]
    x = wl.make_inputs(w, device="cuda", with_dO=False)
    S = dsv.predict_scores(x.Q, x.K, x.Wq, x.Wk, w.block)
    ref = [t.clone() for t in dsv.topk_blocks(S, x.k_per_head, w.block, w.N, w.d)]
    B, H, G, nb = S.shape
    nnz = dsv.nnz_of(B, G, x.k_per_head)
    for _ in range(2):
        outs = (torch.full((B * H * G + 1,), -1, dtype=torch.int32, device="cuda"),
                torch.full((nnz,), -1, dtype=torch.int32, device="cuda"),
                torch.full((B * H * nb + 1,), -1, dtype=torch.int32, device="cuda"),
                torch.full((nnz,), -1, dtype=torch.int32, device="cuda"))
        st = _raw_noalloc(dsv, S, x.k_per_head, w, outs)
        assert st == dsv.DSV_OK, dsv.status_string(st)
        torch.cuda.synchronize()
        assert dsv.device_error()[0] == 0
        for got, want in zip(outs, ref):
            assert torch.equal(got, want)
    # the Python wrapper (its room and dtype checks, then the same entry point)
    outs = tuple(torch.full_like(t, -1) for t in ref)
    dsv.topk_blocks_noalloc(S, x.k_per_head, w.block, w.N, w.d, outs=outs)
    torch.cuda.synchronize()
    for got, want in zip(outs, ref):
        assert torch.equal(got, want)


def test_noalloc_refuses_problems_beyond_its_scratch(dsv):
    w = wl.scaled(wl.WORKLOADS["long518k"], name="too_big", H=64)   # about 130 MiB of top-k scratch
    B, H, G = w.B, w.H, w.nb
    assert dsv.topk_workspace_bytes(B, H, w.N, w.d, w.block) > (64 << 20)
    fake = 1 << 20                                                   # never dereferenced: refused on the host
    karr = (ctypes.c_int32 * H)(*([203] * H))
    st = dsv.lib.dsv_topk_blocks_noalloc(fake, dsv.Shape(B, H, w.N, w.d, w.block, 8), karr,
                                         fake, fake, fake, fake, None)
    assert st == dsv.DSV_ERR_UNSUPPORTED
