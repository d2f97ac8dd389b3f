"""Pins of the oracle's mass-threshold selection (DSV pages, "Technische
samenvatting" 2A and the Hindi summary 2A: the critical KV carries about 90 %
of the attention score), independent of its sort-and-cumsum form."""
import itertools
import math

import numpy as np
import pytest

import oracle


def _brute_m(s, tau, temp):
    # smallest subset size whose best subset carries p-mass >= tau, by enumeration
    p = np.exp(temp * (s - s.max()))
    p = p / p.sum()
    n = len(s)
    for m in range(1, n + 1):
        best = max(sum(p[list(c)]) for c in itertools.combinations(range(n), m))
        if best >= tau:
            return m
    return n


def test_mass_count_brute_force(rng):
    for trial in range(60):
        n = int(rng.integers(1, 8))
        s = rng.normal(size=n) * rng.uniform(0.1, 3.0)
        tau = float(rng.uniform(0.05, 0.99))
        temp = float(rng.uniform(0.2, 4.0))
        m_ref = _brute_m(s, tau, temp)
        assert oracle.mass_count_row(s, tau, temp, 1, n) == m_ref


def test_mass_count_uniform_row_closed_form():
    # equal scores: p_j = 1/nb, so m = ceil(tau * nb) (values chosen exact in binary)
    for nb, tau, m in ((8, 0.75, 6), (16, 0.5, 8), (4, 0.25, 1), (4, 1.0, 4), (32, 0.03125, 1)):
        assert oracle.mass_count_row(np.full(nb, 1.7), tau, 0.8, 1, nb) == m


def test_mass_count_two_levels_closed_form():
    # u blocks at score a, v at score b < a: p_a = e^{ta} / (u e^{ta} + v e^{tb})
    u, v, a, b, t = 3, 5, 2.0, 0.0, 1.0
    pa = math.exp(t * a) / (u * math.exp(t * a) + v * math.exp(t * b))
    pb = math.exp(t * b) / (u * math.exp(t * a) + v * math.exp(t * b))
    s = np.array([b] * v + [a] * u)
    for tau in (0.2, 0.5, 0.8, 0.9, 0.95):
        need_a = math.ceil(tau / pa - 1e-12)
        m = need_a if need_a <= u else u + math.ceil((tau - u * pa) / pb - 1e-12)
        assert oracle.mass_count_row(s, tau, t, 1, u + v) == m


def test_mass_count_limits_and_clamps():
    s = np.array([0.3, 2.0, -1.0, 1.5, 0.9])
    # a very sharp softmax puts all the mass on the unique maximum
    assert oracle.mass_count_row(s, 0.9, 1e3, 1, 5) == 1
    # a very flat one spreads it evenly: ceil(0.9 * 5) = 5
    assert oracle.mass_count_row(s, 0.9, 1e-9, 1, 5) == 5
    # clamps
    assert oracle.mass_count_row(s, 0.9, 1e3, 2, 5) == 2
    assert oracle.mass_count_row(s, 0.9, 1e-9, 1, 3) == 3
    # a non-finite score: kmax
    assert oracle.mass_count_row(np.array([0.1, np.inf, 0.2]), 0.5, 1.0, 1, 2) == 2
    assert oracle.mass_count_row(np.array([0.1, np.nan, 0.2]), 0.5, 1.0, 1, 3) == 3


def test_mass_count_monotone_in_tau(rng):
    s = rng.normal(size=40)
    ms = [oracle.mass_count_row(s, tau, 1.3, 1, 40) for tau in np.linspace(0.01, 1.0, 50)]
    assert all(b >= a for a, b in zip(ms, ms[1:]))
    assert ms[-1] == 40 and ms[0] == 1


def test_mass_lists_are_topk_of_their_own_size(rng):
    S = rng.normal(size=(2, 3, 5, 12))
    S[0, 1, 2, 4] = S[0, 1, 2, 9]             # a tie inside a row
    ptr, col = oracle.mass_lists(S, 0.8, 1.1, 2, 9)
    row = 0
    for b in range(2):
        for h in range(3):
            for g in range(5):
                m = int(ptr[row + 1] - ptr[row])
                assert 2 <= m <= 9 and m == oracle.mass_count_row(S[b, h, g], 0.8, 1.1, 2, 9)
                assert np.array_equal(col[ptr[row]:ptr[row + 1]], oracle.topk_row(S[b, h, g], m))
                row += 1
