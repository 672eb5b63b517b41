"""Pins for the oracle's LM-head confidence (section 3.4.3 'The Core Idea')."""
import json
import math
import os

import numpy as np
import pytest
import scipy.special

from oracle import fdllm_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rows_from_probs(probs):
    # one hidden unit: h = [1], W[:, 0] = log p  ->  logits = log p, softmax = p
    w = np.log(np.asarray(probs, dtype=np.float64))[:, None]
    return np.ones((1, 1)), w


def test_worked_values_from_the_page():
    cases = json.load(open(os.path.join(GOLD, "confidence_worked.json")))["cases"]
    for c in cases:
        h, w = _rows_from_probs(c["probs"])
        st = O.lm_head_confidence(h, w)
        assert st["token"][0] == c["token"]
        assert st["conf"][0] == pytest.approx(c["conf"], abs=1e-12)
        # kappa = log((1 - c) / c)
        assert st["kappa"][0] == pytest.approx(math.log((1 - c["conf"]) / c["conf"]), abs=1e-12)


def test_zero_weights_give_uniform_confidence_and_lowest_index():
    v = 37
    st = O.lm_head_confidence(np.random.default_rng(0).normal(size=(3, 8)), np.zeros((v, 8)))
    assert np.all(st["token"] == 0)
    assert np.allclose(st["conf"], 1.0 / v, rtol=0, atol=1e-15)
    assert np.allclose(st["kappa"], math.log(v - 1), atol=1e-12)


def test_two_token_vocab_is_a_logistic():
    rng = np.random.default_rng(1)
    h = rng.normal(size=(50, 4))
    w = rng.normal(size=(2, 4))
    st = O.lm_head_confidence(h, w)
    l = h @ w.T
    gap = np.abs(l[:, 0] - l[:, 1])
    assert np.allclose(st["conf"], 1.0 / (1.0 + np.exp(-gap)), atol=1e-14)
    assert np.allclose(st["kappa"], -gap, atol=1e-12)
    assert np.array_equal(st["token"], (l[:, 1] > l[:, 0]).astype(int))


def test_against_scipy_softmax_and_logsumexp():
    rng = np.random.default_rng(2)
    h = rng.normal(size=(20, 16))
    w = rng.normal(size=(300, 16)) * 0.7
    st = O.lm_head_confidence(h, w)
    l = h @ w.T
    p = scipy.special.softmax(l, axis=1)
    assert np.allclose(st["conf"], p.max(axis=1), atol=1e-14)
    assert np.array_equal(st["token"], p.argmax(axis=1))
    # kappa = logsumexp over the non-argmax logits minus the max logit
    rest = l.copy()
    rest[np.arange(20), st["token"]] = -np.inf
    assert np.allclose(st["kappa"], scipy.special.logsumexp(rest, axis=1) - l.max(axis=1), atol=1e-12)


def test_kappa_stays_finite_when_confidence_saturates():
    # logits: 0 at index 3, -100 at index 0 and -101.5 elsewhere: c rounds to 1.0 in float64
    mp = pytest.importorskip("mpmath")
    v = 6
    l = np.full(v, -101.5)
    l[3] = 0.0
    l[0] = -100.0
    st = O.lm_head_confidence(np.ones((1, 1)), l[:, None])
    assert st["conf"][0] == 1.0
    mp.mp.dps = 50
    exact = mp.log(mp.e ** -100 + 4 * mp.e ** mp.mpf(-101.5))
    assert st["kappa"][0] == pytest.approx(float(exact), rel=1e-14)
    assert st["token"][0] == 3
    assert st["gap"][0] == 100.0


def test_tie_on_the_max_takes_the_lowest_id():
    l = np.array([1.0, 3.0, 0.5, 3.0, 3.0])
    st = O.lm_head_confidence(np.ones((1, 1)), l[:, None])
    assert st["token"][0] == 1
    assert st["gap"][0] == 0.0
    assert st["conf"][0] == pytest.approx(1 / np.exp(l - 3).sum(), abs=1e-15)


def test_threshold_log_odds_matches_the_confidence_comparison():
    for tau in (0.5, 0.7, 0.9, 0.95, 0.999):
        kt = O.threshold_log_odds(tau)
        for c in (tau - 1e-9, tau + 1e-9, 0.3, 0.999999):
            kappa = math.log((1 - c) / c)
            assert (kappa < kt) == (c > tau)
    assert O.threshold_log_odds(1.0) == -math.inf
