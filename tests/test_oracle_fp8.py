"""Pins of the oracle's FP8 (E4M3) weight-cache functions against things other than
themselves: torch's float8_e4m3fn (an independent library conversion), brute force
over the 253 finite E4M3 values, hand-checked values of the format, and exact
identities of the per-row scale."""
import math

import numpy as np
import pytest
import torch

from oracle import fdllm_oracle as O

FINITE = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def test_decode_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours, ref = O.e4m3_decode(codes), torch_decode(codes)
    nan = np.isnan(ref)
    assert nan.sum() == 2 and np.all(np.isnan(ours[nan]))
    assert np.array_equal(ours[~nan], ref[~nan])


@pytest.mark.parametrize("code,value", [(0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6),
                                        (0x38, 1.0), (0x39, 1.125), (0x3F, 1.875), (0x40, 2.0), (0x7E, 448.0),
                                        (0xB8, -1.0), (0xFE, -448.0)])
def test_decode_hand_values(code, value):
    assert O.e4m3_decode(np.array([code]))[0] == value


def test_encode_inverts_decode():
    vals = O.e4m3_decode(FINITE)
    assert np.array_equal(O.e4m3_encode(vals), FINITE)


@pytest.mark.parametrize("y,want", [(1.0625, 1.0), (1.1875, 1.25), (2.0 ** -10, 0.0), (3 * 2.0 ** -10, 2.0 ** -8),
                                    (2.5 * 2.0 ** -9, 2 * 2.0 ** -9), (3.5 * 2.0 ** -9, 4 * 2.0 ** -9),
                                    (440.0, 448.0), (432.0, 448.0), (424.0, 416.0), (-17.0, -16.0), (-19.0, -20.0),
                                    (0.0146484375, 0.015625)])
def test_round_ties_to_even_hand_values(y, want):
    # midpoints go to the neighbour with an even mantissa: 1 + 1/16 -> 1, 1 + 3/16 -> 1.25; 432 is
    # the midpoint of 416 (mantissa 5) and 448 (6); 17 of 16 (0) and 18 (1); 19 of 18 (1) and 20 (2);
    # 424 is nearer 416
    assert O.e4m3_round(np.array([y]))[0] == want


def test_round_is_the_nearest_value_by_brute_force():
    grid = O.e4m3_decode(FINITE)
    rng = np.random.default_rng(1)
    y = (rng.standard_normal(3000) * np.exp2(rng.integers(-12, 9, 3000))).astype(np.float32).astype(np.float64)
    y = np.clip(y, -448, 448)
    # add exact midpoints of neighbouring grid values
    pos = np.unique(grid[grid >= 0])
    y = np.concatenate([y, (pos[:-1] + pos[1:]) / 2, -(pos[:-1] + pos[1:]) / 2])
    got = O.e4m3_round(y)
    for yi, gi in zip(y, got):
        d = np.abs(grid - yi)
        best = grid[d == d.min()]
        if len(best) == 1:
            assert gi == best[0], (yi, gi, best)
        else:                                   # a tie: the value whose code has an even mantissa
            codes = O.e4m3_encode(np.unique(best))
            even = [O.e4m3_decode(np.array([c]))[0] for c in codes if (c & 1) == 0]
            assert gi in even, (yi, gi, best)


def test_round_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(2)
    y = (rng.standard_normal(200000) * np.exp2(rng.integers(-16, 9, 200000))).astype(np.float32)
    y = np.clip(y, -448, 448).astype(np.float64)
    assert np.array_equal(O.e4m3_round(y), torch.from_numpy(y).to(torch.float8_e4m3fn).double().numpy())


def test_round_codes_match_torch_including_signed_zero():
    """Byte codes, not values: a negative input that rounds to zero gives -0 (0x80), as IEEE
    rounding keeps the operand's sign."""
    rng = np.random.default_rng(8)
    y = (rng.standard_normal(20000) * np.exp2(rng.integers(-14, 9, 20000))).astype(np.float32)
    y = np.concatenate([np.clip(y, -448, 448), np.array([-0.0, 0.0, -1e-5, 1e-5, -2.0 ** -10, 2.0 ** -10],
                                                         dtype=np.float32)]).astype(np.float64)
    ours = O.e4m3_encode(O.e4m3_round(y))
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)
    assert ours[-6] == 0x80 and ours[-5] == 0x00 and ours[-4] == 0x80


@pytest.mark.parametrize("amax,k", [(448.0, 0), (np.nextafter(448.0, 1e9), 1), (224.0, -1), (224.5, 0),
                                    (1.0, -8), (0.0, 0), (896.0, 1), (897.0, 2), (2.0 ** -20, -28)])
def test_scale_exponent_hand_values(amax, k):
    assert O.fp8_scale_exponent(amax) == k


def test_scale_exponent_is_the_smallest_that_fits():
    rng = np.random.default_rng(3)
    for amax in np.exp2(rng.uniform(-30, 30, 2000)):
        k = O.fp8_scale_exponent(amax)
        assert amax <= 448.0 * 2.0 ** k and amax > 448.0 * 2.0 ** (k - 1)


def test_quantized_rows_use_the_top_binade_and_round_within_half_a_step():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((6, 300)) * np.array([1e-3, 0.05, 1.0, 7.0, 300.0, 5e4])[:, None]).astype(np.float32)
    codes, scales = O.quantize_fp8_rows(x)
    deq = O.dequantize_fp8_rows(codes, scales)
    for r in range(x.shape[0]):
        q = np.abs(O.e4m3_decode(codes[r]))
        assert 224.0 <= q.max() <= 448.0               # the scale puts the row maximum in the top binade
        assert math.log2(scales[r]).is_integer()
        # round to nearest: within half a grid step (relative 2^-4 for normal values, 2^-10 absolute below)
        err = np.abs(deq[r] - x[r]) / scales[r]
        tol = np.maximum(np.abs(x[r]) / scales[r] * 2.0 ** -4, 2.0 ** -10)
        assert np.all(err <= tol)
    z_codes, z_scales = O.quantize_fp8_rows(np.zeros((1, 8)))
    assert np.all(z_codes == 0) and z_scales[0] == 1.0


def test_fp8_confidence_equals_the_plain_one_on_exactly_representable_operands():
    """Rows already on the E4M3 grid with max |row| = 448 quantise to themselves (scale 1), so the
    FP8 path must give lm_head_confidence of the same values."""
    rng = np.random.default_rng(5)
    grid = O.e4m3_decode(FINITE)
    small = grid[np.abs(grid) <= 2.0]
    h = rng.choice(small, size=(4, 64))
    h[:, 0] = 448.0
    w = rng.choice(small, size=(50, 64))
    w[:, 1] = -448.0
    wc, ws = O.quantize_fp8_rows(w)
    assert np.all(ws == 1.0) and np.array_equal(O.e4m3_decode(wc), w)
    a = O.lm_head_confidence_fp8(h, wc, ws)
    b = O.lm_head_confidence(h, w)
    for key in ("token", "conf", "kappa", "gap"):
        assert np.array_equal(a[key], b[key]), key


def test_fp8_confidence_zero_weight_is_uniform():
    rng = np.random.default_rng(6)
    h = rng.standard_normal((3, 32))
    wc, ws = O.quantize_fp8_rows(np.zeros((10, 32)))
    st = O.lm_head_confidence_fp8(h, wc, ws)
    assert np.allclose(st["conf"], 0.1) and np.all(st["token"] == 0)


def test_fp8_confidence_scales_multiply_the_logits():
    """Scaling W rows by powers of two changes only the scales, so the logits scale exactly."""
    rng = np.random.default_rng(7)
    h = rng.standard_normal((2, 48))
    w = rng.standard_normal((20, 48))
    wc, ws = O.quantize_fp8_rows(w)
    wc2, ws2 = O.quantize_fp8_rows(w * 8.0)
    assert np.array_equal(wc, wc2) and np.array_equal(ws2, ws * 8.0)
    l1 = O.lm_head_confidence_fp8(h, wc, ws)["logits"]
    l2 = O.lm_head_confidence_fp8(h, wc2, ws2)["logits"]
    assert np.array_equal(l2, l1 * 8.0)


def test_kv_rows_quantise_per_position_and_head():
    """Each (sequence, position, head) row gets its own scale: scaling one row by 2^j changes only
    that row's scale, and the window splice leaves every other row's codes and scales alone."""
    rng = np.random.default_rng(9)
    x = rng.standard_normal((2, 6, 3, 16))
    c, s = O.quantize_kv_rows(x)
    assert c.shape == x.shape and s.shape == (2, 6, 3)
    y = x.copy()
    y[1, 4, 2] *= 2.0 ** 5
    c2, s2 = O.quantize_kv_rows(y)
    assert np.array_equal(c2, c) and s2[1, 4, 2] == s[1, 4, 2] * 32
    s2[1, 4, 2] = s[1, 4, 2]
    assert np.array_equal(s2, s)
    src = rng.standard_normal((2, 2, 3, 16)) * 100
    nc, ns = O.kv_splice_fp8(c, s, src, 3)
    keep = np.ones(6, dtype=bool)
    keep[3:5] = False
    assert np.array_equal(nc[:, keep], c[:, keep]) and np.array_equal(ns[:, keep], s[:, keep])
    deq = O.dequantize_kv_rows(nc, ns)[:, 3:5]
    assert np.all(np.abs(deq - src) <= np.abs(src) * 2.0 ** -4 + ns[:, 3:5, :, None] * 2.0 ** -10)


def test_attention_over_an_exact_fp8_cache_is_the_plain_attention():
    """A cache whose rows are already E4M3 values times powers of two quantises to itself, so the
    attention over the dequantised cache equals the plain block attention."""
    rng = np.random.default_rng(10)
    grid = O.e4m3_decode(FINITE)
    small = grid[np.abs(grid) <= 4.0]
    b, n, hkv, d, s, e = 1, 40, 2, 16, 16, 24
    kc = rng.choice(small, size=(b, n, hkv, d)) * 2.0 ** rng.integers(-3, 3, (b, n, hkv, 1))
    vc = rng.choice(small, size=(b, n, hkv, d)) * 2.0 ** rng.integers(-3, 3, (b, n, hkv, 1))
    kc[..., 0] = 448.0 * 2.0 ** -7                  # every row's maximum sets its scale to 2^-7 ...
    vc[..., 0] = 448.0 * 2.0 ** -7
    kc[..., 1:] = np.clip(kc[..., 1:], -2.0, 2.0)   # ... and every value is a grid value at that scale
    vc[..., 1:] = np.clip(vc[..., 1:], -2.0, 2.0)
    kq, ks = O.quantize_kv_rows(kc)
    vq, vs = O.quantize_kv_rows(vc)
    assert np.array_equal(O.dequantize_kv_rows(kq, ks), kc) and np.array_equal(O.dequantize_kv_rows(vq, vs), vc)
    q = rng.standard_normal((b, e - s, 4, d))
    kf = rng.standard_normal((b, e - s, hkv, d))
    vf = rng.standard_normal((b, e - s, hkv, d))
    a = O.block_attention(q, O.dequantize_kv_rows(kq, ks), O.dequantize_kv_rows(vq, vs), kf, vf, mode="dual", s=s,
                          e=e, n_q_heads=4, n_kv_heads=hkv)
    r = O.block_attention(q, kc, vc, kf, vf, mode="dual", s=s, e=e, n_q_heads=4, n_kv_heads=hkv)
    assert np.array_equal(a[0], r[0]) and np.array_equal(a[1], r[1])
