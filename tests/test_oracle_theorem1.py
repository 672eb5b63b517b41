"""Theorem 1 (section 3.4.3) by brute force over tiny vocabularies.

If every position's marginal puts more than 1 - eps on x*_j and (n + 1) eps <= 1,
the greedy (argmax) choice under the product of marginals equals the greedy
choice under the joint and both equal x*; the bound is tight (the page's
counterexample).  The distance bounds are checked on the same tables."""
import itertools
import math

import numpy as np
import pytest

from oracle import fdllm_oracle as O


def _random_joint_with_confident_marginals(rng, n, v, eps):
    """A joint over V^n whose marginals all exceed 1 - eps at x* = (0, ..., 0)."""
    while True:
        p = rng.dirichlet(np.full(v ** n, 0.3)).reshape((v,) * n)
        # put at least 1 - n * eps * u on x* and spread the rest
        keep = 1.0 - rng.uniform(0.0, 1.0) * eps
        p = p * (1 - keep)
        p[(0,) * n] += keep
        margs = O.marginals(p)
        if all(m[0] > 1 - eps for m in margs):
            return p


@pytest.mark.parametrize("n,v", [(1, 2), (2, 2), (2, 3), (3, 2), (3, 3), (4, 2), (2, 4)])
def test_greedy_equivalence_when_n_plus_one_eps_at_most_one(n, v):
    rng = np.random.default_rng(n * 10 + v)
    eps = 1.0 / (n + 1)
    for _ in range(60):
        p = _random_joint_with_confident_marginals(rng, n, v, eps * rng.uniform(0.2, 1.0))
        q = O.product_of_marginals(p)
        assert O.greedy(p) == (0,) * n
        assert O.greedy(q) == (0,) * n


@pytest.mark.parametrize("n", [2, 3, 4])
def test_tightness_counterexample(n):
    """Above eps = 1/(n+1) the joint's argmax can leave x*, while q's stays there."""
    v = 2
    delta = 0.01
    p = np.zeros((v,) * n)
    # mass 1/(n+1) + delta on each sequence differing from x* in one position; the rest on x*
    for j in range(n):
        z = [0] * n
        z[j] = 1
        p[tuple(z)] = 1.0 / (n + 1) + delta
    p[(0,) * n] = 1.0 - p.sum()
    assert p[(0,) * n] > 0
    eps = max(1 - m[0] for m in O.marginals(p)) + 1e-12
    assert (n + 1) * eps > 1                                 # condition violated
    assert all(m[0] > 1 - eps for m in O.marginals(p))
    assert O.greedy(p) != (0,) * n
    assert O.greedy(O.product_of_marginals(p)) == (0,) * n


@pytest.mark.parametrize("n,v", [(1, 3), (2, 2), (2, 3), (3, 2), (3, 3)])
def test_distance_bounds(n, v):
    rng = np.random.default_rng(100 + n * 10 + v)
    for _ in range(60):
        eps = rng.uniform(0.01, 0.3)
        p = _random_joint_with_confident_marginals(rng, n, v, eps)
        q = O.product_of_marginals(p)
        tv = 0.5 * np.abs(p - q).sum()
        assert tv < (3 * n - 1) / 2 * eps + 1e-15
        mask = p > 0
        kl = float((p[mask] * np.log(p[mask] / q[mask])).sum())
        hb = -eps * math.log(eps) - (1 - eps) * math.log(1 - eps)
        bound = (n - 1) * (hb + eps * math.log(v - 1)) if v > 1 else 0.0
        assert kl <= bound + 1e-12                           # n = 1: both sides are 0


def test_marginals_and_product_by_enumeration():
    rng = np.random.default_rng(7)
    p = rng.dirichlet(np.ones(12)).reshape(2, 3, 2)
    q = O.product_of_marginals(p)
    for x in itertools.product(range(2), range(3), range(2)):
        m0 = sum(p[x[0], a, b] for a in range(3) for b in range(2))
        m1 = sum(p[a, x[1], b] for a in range(2) for b in range(2))
        m2 = sum(p[a, b, x[2]] for a in range(2) for b in range(3))
        assert q[x] == pytest.approx(m0 * m1 * m2, abs=1e-15)
