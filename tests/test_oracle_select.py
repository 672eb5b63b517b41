"""Pins for the oracle's selection rules (section 3.4.3 threshold and factor strategies)."""
import json
import math
import os

import numpy as np
import pytest

from oracle import fdllm_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _kappa(c):
    c = np.asarray(c, dtype=np.float64)
    return np.log((1 - c) / c)


def test_threshold_unmasks_exactly_the_confident_masked_positions():
    conf = np.array([0.95, 0.2, 0.91, 0.99, 0.5, 0.9])
    masked = np.array([True, True, True, False, True, True])
    sel = O.threshold_select(conf, _kappa(conf), masked, 0.9)
    # 0.99 is not masked; 0.9 is not above 0.9 (strict reading)
    assert sel.tolist() == [True, False, True, False, False, False]


def test_fallback_picks_the_single_most_confident_masked_position():
    conf = np.array([0.3, 0.6, 0.6, 0.95, 0.1])
    masked = np.array([True, True, True, False, True])
    sel = O.threshold_select(conf, _kappa(conf), masked, 0.9)
    assert sel.tolist() == [False, True, False, False, False]   # tie at 0.6 -> lowest position
    assert not O.threshold_select(conf, _kappa(conf), np.zeros(5, bool), 0.9).any()


def test_tau_at_least_one_gives_one_token_per_step():
    rng = np.random.default_rng(0)
    for _ in range(200):
        c = rng.uniform(0.01, 1.0, size=12)
        c[rng.integers(0, 12)] = 1.0
        m = rng.random(12) < 0.6
        if not m.any():
            continue
        for tau in (1.0, 1.5):
            sel = O.threshold_select(c, _kappa(np.minimum(c, 1 - 1e-16)), m, tau)
            assert sel.sum() == 1 and m[np.argmax(sel)]


def test_threshold_selection_is_monotone_in_tau():
    rng = np.random.default_rng(1)
    for _ in range(100):
        c = rng.uniform(0.0, 1.0, size=16)
        m = rng.random(16) < 0.7
        prev = None
        for tau in (0.5, 0.7, 0.8, 0.9, 0.95):
            sel = O.threshold_select(c, _kappa(c), m, tau)
            assert sel.sum() >= (1 if m.any() else 0)
            assert not (sel & ~m).any()
            if prev is not None and sel.sum() > 1:
                assert not (sel & ~prev).any()
            prev = sel


def test_factor_rule_on_a_hand_worked_case():
    # (n + 1) (1 - c_(n)) for c sorted = 0.99, 0.95, 0.9, 0.6: 0.02, 0.15, 0.4, 2.0
    c = np.array([0.6, 0.99, 0.9, 0.95])
    m = np.ones(4, bool)
    assert O.factor_select(_kappa(c), m, 1.0).tolist() == [False, True, True, True]
    assert O.factor_select(_kappa(c), m, 0.1).tolist() == [False, True, False, False]
    # even n = 1 fails: 2 * 0.01 = 0.02 >= 0.01 -> still one token
    assert O.factor_select(_kappa(c), m, 0.01).tolist() == [False, True, False, False]
    assert O.factor_select(_kappa(c), m, 2.5).tolist() == [True, True, True, True]


def test_threshold_boundary_arithmetic_from_the_page():
    g = json.load(open(os.path.join(GOLD, "page_arithmetic.json")))["threshold_boundary"]
    eps = 1 - g["tau"]
    assert (g["n"] + 1) * eps == pytest.approx(g["product"], abs=1e-12)


def test_topk_takes_the_k_most_confident():
    c = np.array([0.5, 0.8, 0.3, 0.9, 0.7])
    m = np.array([True, True, True, False, True])
    assert O.topk_select(_kappa(c), m, 2).tolist() == [False, True, False, False, True]
    assert O.topk_select(_kappa(c), m, 10).sum() == 4


def test_block_window_matches_the_page():
    g = json.load(open(os.path.join(GOLD, "page_arithmetic.json")))["block_window"]
    for k1, s, e in g["windows_1based"]:
        assert O.block_window(g["prompt_len"], g["block_size"], k1 - 1) == (s, e)


def test_kv_memory_estimate_from_the_page():
    g = json.load(open(os.path.join(GOLD, "page_arithmetic.json")))["kv_memory"]
    by = O.kv_cache_bytes(g["seq_len"], g["layers"], g["heads"], g["head_dim"], g["bytes_per_elem"])
    assert by == 536_870_912
    assert round(by / 1e6) == 537 and abs(by / 1e6 - g["approx_mb"]) < 1.0
