"""The parity contract's unmask rule (tests/gpu_helpers.compare_select) on hand-made
GPU results, on the CPU: a decision may differ from the oracle's only where the
contract exempts it (|c - tau| < 2e-3, a factor comparison inside the same band,
a near tie of kappa in a ranking or in the fallback), and a wrong decision
elsewhere must fail even when a neighbouring position is inside a band."""
import math

import numpy as np
import pytest

from gpu_helpers import compare_select


def _kappa(c):
    return math.log((1.0 - c) / c)


def _info(conf, unmask, masked=None):
    conf = np.asarray(conf, dtype=np.float64)[None, :]
    B = conf.shape[1]
    masked = np.ones((1, B), dtype=bool) if masked is None else np.asarray(masked, dtype=bool)[None, :]
    kap = np.array([[_kappa(c) for c in conf[0]]])
    return {"masked_before": masked, "conf": np.where(masked, conf, np.nan), "kappa": np.where(masked, kap, np.nan),
            "token": np.where(masked, np.arange(B)[None, :] + 10, -1), "gap": np.full((1, B), 1.0),
            "unmask": np.asarray(unmask, dtype=bool)[None, :]}


def _got(info, unmask):
    m = info["masked_before"]
    return {"unmask": np.asarray(unmask, dtype=bool)[None, :], "conf": np.where(m, info["conf"], np.nan),
            "kappa": np.where(m, info["kappa"], np.nan), "token": info["token"].copy()}


# threshold, tau = 0.9: position 1 sits inside the band (|c - tau| < 2e-3)
CONF = [0.99, 0.8991, 0.5, 0.2]
ORACLE = [True, False, False, False]


def test_threshold_equal_and_band_flip_pass():
    ref = _info(CONF, ORACLE)
    assert compare_select(ref, _got(ref, ORACLE), 0.9) == 0
    assert compare_select(ref, _got(ref, [True, True, False, False]), 0.9) == 1


def test_threshold_confident_position_left_masked_fails():
    """c = 0.99 not selected while a neighbour is in the band: must fail."""
    ref = _info(CONF, ORACLE)
    with pytest.raises(AssertionError):
        compare_select(ref, _got(ref, [False, True, False, False]), 0.9)
    with pytest.raises(AssertionError):
        compare_select(ref, _got(ref, [False, False, False, False]), 0.9)


def test_threshold_position_below_the_band_selected_fails():
    ref = _info(CONF, ORACLE)
    with pytest.raises(AssertionError):
        compare_select(ref, _got(ref, [True, False, True, False]), 0.9)


def test_threshold_fallback_near_tie_passes_and_far_pick_fails():
    conf = [0.60, 0.6000001, 0.3, 0.1]           # nothing above tau: the single most confident
    ref = _info(conf, [False, True, False, False])
    assert compare_select(ref, _got(ref, [True, False, False, False]), 0.9) == 2
    with pytest.raises(AssertionError):
        compare_select(ref, _got(ref, [False, False, True, False]), 0.9)
    with pytest.raises(AssertionError):                 # the fallback unmasks exactly one
        compare_select(ref, _got(ref, [True, True, False, False]), 0.9)


def test_threshold_band_position_decides_fallback():
    """The only near-tau position decides between 'one above tau' and 'fall back': either side
    is valid, but the fallback must then pick a most confident position."""
    conf = [0.9005, 0.7, 0.3]
    ref = _info(conf, [True, False, False])
    assert compare_select(ref, _got(ref, [True, False, False]), 0.9) == 0
    with pytest.raises(AssertionError):
        compare_select(ref, _got(ref, [False, True, False]), 0.9)


def test_unmasking_a_decoded_position_fails():
    ref = _info([0.99, 0.5, 0.4], [True, False, False], masked=[True, False, True])
    with pytest.raises(AssertionError):
        compare_select(ref, _got(ref, [True, True, False]), 0.9)


def test_factor_band_and_prefix():
    # eps = 1 - c: (n + 1) eps_(n) = 2 * 0.01, 3 * 0.3331 = 0.9993 (inside the band around f = 1), 4 * 0.5
    conf = [0.99, 0.6669, 0.5]
    ref = _info(conf, [True, True, False])           # the oracle takes n = 2 (0.9993 < 1)
    assert compare_select(ref, _got(ref, [True, True, False]), 0.9, "factor", 1.0) == 0
    assert compare_select(ref, _got(ref, [True, False, False]), 0.9, "factor", 1.0) == 1
    with pytest.raises(AssertionError):                 # not a most-confident prefix
        compare_select(ref, _got(ref, [False, True, False]), 0.9, "factor", 1.0)
    with pytest.raises(AssertionError):                 # n = 3: 4 * 0.5 = 2, far outside the band
        compare_select(ref, _got(ref, [True, True, True]), 0.9, "factor", 1.0)


def test_factor_count_outside_band_fails():
    conf = [0.999, 0.99, 0.6]                          # 2 * 0.001, 3 * 0.01 < 1; 4 * 0.4 > 1 (far)
    ref = _info(conf, [True, True, False])
    with pytest.raises(AssertionError):
        compare_select(ref, _got(ref, [True, False, False]), 0.9, "factor", 1.0)


def test_topk_near_tie_passes_and_wrong_count_fails():
    conf = [0.7, 0.70000001, 0.2]
    ref = _info(conf, [False, True, False])
    assert compare_select(ref, _got(ref, [True, False, False]), 0.9, "topk") == 2
    with pytest.raises(AssertionError):
        compare_select(ref, _got(ref, [True, True, False]), 0.9, "topk")
    with pytest.raises(AssertionError):
        compare_select(ref, _got(ref, [False, False, True]), 0.9, "topk")
