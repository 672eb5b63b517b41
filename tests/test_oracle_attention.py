"""Pins for the oracle's block attention (section 3.4.2 PrefixCache / DualCache)."""
import math

import numpy as np
import pytest
import torch

from oracle import fdllm_oracle as O


def _rand(rng, *shape):
    return rng.normal(size=shape)


def test_full_attention_matches_torch_sdpa_with_gqa():
    rng = np.random.default_rng(0)
    b, nq, n, hq, hkv, d = 2, 5, 17, 6, 2, 16
    q, k, v = _rand(rng, b, nq, hq, d), _rand(rng, b, n, hkv, d), _rand(rng, b, n, hkv, d)
    o, lse = O.attention_full(q, k, v, hq, hkv)
    tq = torch.from_numpy(q).permute(0, 2, 1, 3)
    tk = torch.from_numpy(k).permute(0, 2, 1, 3).repeat_interleave(hq // hkv, dim=1)
    tv = torch.from_numpy(v).permute(0, 2, 1, 3).repeat_interleave(hq // hkv, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv).permute(0, 2, 1, 3).numpy()
    assert np.allclose(o, ref, atol=1e-12)
    scores = torch.einsum("bhqd,bhkd->bhqk", tq, tk) / math.sqrt(d)
    assert np.allclose(lse, torch.logsumexp(scores, dim=-1).permute(0, 2, 1).numpy(), atol=1e-12)


def test_single_key_returns_its_value_and_equal_scores_average():
    rng = np.random.default_rng(1)
    q, k, v = _rand(rng, 1, 3, 2, 8), _rand(rng, 1, 1, 2, 8), _rand(rng, 1, 1, 2, 8)
    o, lse = O.attention_full(q, k, v, 2, 2)
    assert np.allclose(o, np.broadcast_to(v, o.shape), atol=1e-15)
    # q = 0: every score is 0 -> output is the mean of V, lse = log N
    n = 9
    v = _rand(rng, 1, n, 1, 8)
    o, lse = O.attention_full(np.zeros((1, 2, 1, 8)), _rand(rng, 1, n, 1, 8), v, 1, 1)
    assert np.allclose(o[0, :, 0], v[0, :, 0].mean(axis=0), atol=1e-14)
    assert np.allclose(lse, math.log(n), atol=1e-14)


def test_two_keys_closed_form():
    d = 4
    q = np.zeros((1, 1, 1, d)); q[0, 0, 0, 0] = 2.0
    k = np.zeros((1, 2, 1, d)); k[0, 0, 0, 0] = 1.0; k[0, 1, 0, 0] = -1.0
    v = np.zeros((1, 2, 1, d)); v[0, 0, 0, 1] = 3.0; v[0, 1, 0, 2] = 5.0
    o, _ = O.attention_full(q, k, v, 1, 1)
    a = 2.0 / math.sqrt(d)                  # the two scores are +a and -a
    w0 = 1.0 / (1.0 + math.exp(-2 * a))
    assert o[0, 0, 0, 1] == pytest.approx(3.0 * w0, abs=1e-15)
    assert o[0, 0, 0, 2] == pytest.approx(5.0 * (1 - w0), abs=1e-15)


@pytest.mark.parametrize("mode", ["dual", "prefix", "none"])
def test_refresh_every_step_equals_full_attention(mode):
    """With the cache refreshed at every step (cache == this step's K/V), the cached
    step equals full bidirectional attention over the whole sequence, on the query rows."""
    rng = np.random.default_rng(2)
    b, p, bs, nblk, hq, hkv, d = 2, 12, 4, 3, 4, 2, 8
    n = p + bs * nblk
    q_all, k_all, v_all = _rand(rng, b, n, hq, d), _rand(rng, b, n, hkv, d), _rand(rng, b, n, hkv, d)
    full_o, full_lse = O.attention_full(q_all, k_all, v_all, hq, hkv)
    for blk in range(nblk):
        s, e = O.block_window(p, bs, blk)
        pos = O.query_positions(mode, s, e, n)
        sl = slice(pos.start, pos.stop)
        o, lse = O.block_attention(q_all[:, sl], k_all, v_all, k_all[:, sl], v_all[:, sl],
                                   mode=mode, s=s, e=e, n_q_heads=hq, n_kv_heads=hkv)
        assert np.allclose(o, full_o[:, sl], atol=1e-12)
        assert np.allclose(lse, full_lse[:, sl], atol=1e-12)


def test_cache_positions_are_read_from_the_right_source():
    """DualCache reads prefix and suffix from the cache and the block from the fresh K/V."""
    rng = np.random.default_rng(3)
    b, n, hkv, d = 1, 20, 1, 4
    s, e = 8, 12
    kc, vc = _rand(rng, b, n, hkv, d), _rand(rng, b, n, hkv, d)
    kf, vf = _rand(rng, b, e - s, hkv, d), _rand(rng, b, e - s, hkv, d)
    q = _rand(rng, b, e - s, 1, d)
    base, _ = O.block_attention(q, kc, vc, kf, vf, mode="dual", s=s, e=e, n_q_heads=1, n_kv_heads=1)
    kc2 = kc.copy(); kc2[:, s:e] += 10.0          # cache rows inside the window are never read
    same, _ = O.block_attention(q, kc2, vc, kf, vf, mode="dual", s=s, e=e, n_q_heads=1, n_kv_heads=1)
    assert np.array_equal(base, same)
    for rows in (slice(0, s), slice(e, n)):       # prefix and suffix cache rows are read
        vc3 = vc.copy(); vc3[:, rows] += 1.0
        diff, _ = O.block_attention(q, kc, vc3, kf, vf, mode="dual", s=s, e=e, n_q_heads=1, n_kv_heads=1)
        assert not np.allclose(base, diff)
    # PrefixCache: the suffix comes from the fresh projections, so its cache rows are not read
    kf_p, vf_p = _rand(rng, b, n - s, hkv, d), _rand(rng, b, n - s, hkv, d)
    qp = _rand(rng, b, n - s, 1, d)
    bp, _ = O.block_attention(qp, kc, vc, kf_p, vf_p, mode="prefix", s=s, e=e, n_q_heads=1, n_kv_heads=1)
    vc4 = vc.copy(); vc4[:, e:] += 5.0
    sp, _ = O.block_attention(qp, kc, vc4, kf_p, vf_p, mode="prefix", s=s, e=e, n_q_heads=1, n_kv_heads=1)
    assert np.array_equal(bp, sp)


def test_splice_writes_exactly_the_window():
    rng = np.random.default_rng(4)
    cache = _rand(rng, 2, 10, 2, 4)
    src = _rand(rng, 2, 3, 2, 4)
    out = O.kv_splice(cache, src, 5)
    assert np.array_equal(out[:, 5:8], src)
    assert np.array_equal(out[:, :5], cache[:, :5]) and np.array_equal(out[:, 8:], cache[:, 8:])
