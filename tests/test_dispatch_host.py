"""The OP dispatcher (dsv_dispatch_heads), host-only: its decisions against
the stated rule, and its argument checks (CPU, no GPU needed)."""
import math

import numpy as np
import pytest


@pytest.fixture(scope="module")
def dsv():
    from dynamic_block_sparse_projection_gb300.build import build
    build()
    from dynamic_block_sparse_projection_gb300 import binding
    return binding


def _rule(k, nb, rho, ratio):
    """Dense when the profile's sparse/dense time ratio at rho = k / nb,
    piecewise linear between points and constant beyond the ends, is >= 1."""
    x = k / nb
    if x <= rho[0]:
        y = ratio[0]
    elif x >= rho[-1]:
        y = ratio[-1]
    else:
        i = next(i for i in range(1, len(rho)) if rho[i] >= x)
        t = (x - rho[i - 1]) / (rho[i] - rho[i - 1])
        y = ratio[i - 1] + t * (ratio[i] - ratio[i - 1])
    return y >= 1.0


def test_dispatch_follows_the_rule_on_random_profiles(dsv):
    rng = np.random.default_rng(3)
    for _ in range(200):
        n = int(rng.integers(1, 8))
        rho = np.sort(rng.choice(np.arange(1, 101), size=n, replace=False)) / 100.0
        ratio = rng.uniform(0.2, 1.8, size=n)
        nb = int(rng.integers(1, 300))
        ks = [int(v) for v in rng.integers(1, nb + 1, size=int(rng.integers(1, 9)))]
        k_out, dense = dsv.dispatch_heads(ks, nb, rho.astype(np.float32), ratio.astype(np.float32))
        for k, ko, de in zip(ks, k_out, dense):
            want = _rule(k, nb, rho.astype(np.float32).astype(np.float64), ratio.astype(np.float32).astype(np.float64))
            assert de == want, (k, nb, rho, ratio)
            assert ko == (nb if want else k)


def test_dispatch_edges(dsv):
    # one point: a constant profile
    assert dsv.dispatch_heads([3, 7], 10, [0.5], [0.9]) == ([3, 7], [False, False])
    assert dsv.dispatch_heads([3, 7], 10, [0.5], [1.0]) == ([10, 10], [True, True])
    # the crossover itself goes dense; beyond the ends the end values hold
    assert dsv.dispatch_heads([5], 10, [0.25, 0.75], [0.5, 1.5]) == ([10], [True])
    assert dsv.dispatch_heads([1, 90], 100, [0.2, 0.8], [0.3, 1.2]) == ([1, 100], [False, True])
    # k = nb: ratio at rho = 1
    assert dsv.dispatch_heads([64], 64, [0.1, 1.0], [0.2, 0.99]) == ([64], [False])


@pytest.mark.parametrize("args", [
    ([3], 10, [0.5, 0.5], [0.9, 1.1]),          # rho not increasing
    ([3], 10, [0.0, 0.5], [0.9, 1.1]),          # rho outside (0, 1]
    ([3], 10, [0.5, 1.5], [0.9, 1.1]),
    ([3], 10, [0.5], [0.0]),                    # ratio not > 0
    ([3], 10, [0.5], [math.nan]),
    ([3], 10, [0.5], [math.inf]),
    ([0], 10, [0.5], [0.9]),                    # k outside [1, nb]
    ([11], 10, [0.5], [0.9]),
    ([3], 10, [], []),                          # empty profile
])
def test_dispatch_rejects_bad_arguments(dsv, args):
    with pytest.raises(dsv.DsvError) as e:
        dsv.dispatch_heads(*args)
    assert e.value.status == dsv.DSV_ERR_INVALID_ARG
