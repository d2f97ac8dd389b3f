import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def to_np64(t):
    """torch tensor (any dtype, any device) -> float64 numpy array on the host."""
    import torch
    return t.detach().to("cpu", torch.float64).numpy()


def rel_l2(x, y):
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    den = np.linalg.norm(y.ravel())
    return float(np.linalg.norm((x - y).ravel()) / (den if den > 0 else 1.0))


@pytest.fixture
def rng():
    return np.random.default_rng(12345)
