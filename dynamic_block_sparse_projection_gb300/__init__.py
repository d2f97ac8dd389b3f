"""DSV dynamic sparse 3D attention on GB300 (sm_103a).

Four C-ABI calls in ``libdsv.so`` form the hot path: dsv_predict_scores,
dsv_topk_blocks, dsv_sparse_attn_fwd and dsv_sparse_attn_bwd.  The Python
binding in :mod:`.binding` only marshals arguments; submodules load lazily so
that the seeded workload generator in :mod:`.workloads` can be used without
the CUDA library.
"""
import importlib

__all__ = ["workloads", "binding"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
