"""The shared seeded input generator: determinism, exactness and distribution."""
import numpy as np
import pytest
import torch

from block_cached_decoding_gb300 import synth


def test_splitmix_reference_values():
    # SplitMix64 seeded with 0: the published first outputs of the generator
    out = [int(synth.splitmix(np.uint64(0), i)) for i in range(3)]
    assert out == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_normals_are_exact_multiples_and_reproducible():
    k = synth.stream_key(5, synth.KIND_W)
    a = synth.normal12_f32(k, 1000)
    b = synth.normal12_f32(k, 400, offset=600)
    assert np.array_equal(a[600:], b)
    assert np.all(a * 65536 == np.round(a * 65536))
    big = synth.normal12_f32(synth.stream_key(6, 2), 400_000)
    assert abs(big.mean()) < 0.01 and abs(big.var() - 1) < 0.01
    assert np.abs(big).max() <= 6.0


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = (rng.normal(size=100_000) * rng.choice([1e-3, 1, 1e3], 100_000)).astype(np.float32)
    x[:4] = [1.00390625, 1.01171875, -1.00390625, 3.0]     # exact halfway cases
    ours = synth.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_streams_differ_across_coordinates():
    a = synth.per_position(1, synth.KIND_Q, 2, 0, [3, 4], 16, "f32")
    assert not np.array_equal(a[0, 0], a[0, 1]) and not np.array_equal(a[0, 0], a[1, 0])
    b = synth.per_position(1, synth.KIND_Q, 2, 1, [3, 4], 16, "f32")
    assert not np.array_equal(a, b)
    assert synth.stream_key(1, 0, 5) != synth.stream_key(1, 5)


def test_plant_rate_and_target_range():
    planted, target = synth.plant_draws(3, 4, 0, range(500), 0.4, 126464)
    assert abs(planted.mean() - 0.4) < 0.05
    assert target.min() >= 0 and target.max() < 126464


def test_lm_head_row_matches_the_full_weight():
    w = synth.lm_head_weight(9, 50, 32, 0.1, "bf16")
    assert np.array_equal(synth.lm_head_row(9, 17, 32, 0.1, "bf16"), w[17])
