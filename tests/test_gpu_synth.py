"""The device twin of the seeded generator produces the host generator's bytes."""
import numpy as np
import pytest
import torch

from block_cached_decoding_gb300 import fdllm as F
from block_cached_decoding_gb300 import synth
from gpu_helpers import dev, ensure_built, tdtype

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.cpu().numpy()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_weight_and_cache_streams(dtype):
    V, H = 300, 128
    w = torch.empty(V, H, dtype=tdtype(dtype), device="cuda")
    F.fdllm_synth_normals(7, F.SYNTH_W, [], V * H, 0, 0.1414, F.F32 if dtype == "f32" else F.BF16, w)
    assert np.array_equal(_bits(w), synth.lm_head_weight(7, V, H, 0.1414, dtype))
    kc = torch.empty(2, 40, 2, 64, dtype=tdtype(dtype), device="cuda")
    F.fdllm_synth_kv_cache(7, F.SYNTH_KCACHE, 2, 40, 2, 64, 3, 1.0, F.F32 if dtype == "f32" else F.BF16, kc)
    assert np.array_equal(_bits(kc), synth.kv_cache(7, synth.KIND_KCACHE, 2, 40, 2, 64, 3, dtype))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rows_hidden_and_prompt(dtype):
    dc = F.F32 if dtype == "f32" else F.BF16
    q = torch.empty(3, 5, 4 * 64, dtype=tdtype(dtype), device="cuda")
    F.fdllm_synth_rows(11, F.SYNTH_Q, 3, 2, 70, 5, 4 * 64, 1.0, dc, q)
    assert np.array_equal(_bits(q), synth.per_position(11, synth.KIND_Q, 3, 2, range(70, 75), 256, dtype))
    V, H = 1000, 256
    w_host = synth.lm_head_weight(11, V, H, 0.2236, dtype)
    w = dev(w_host, dtype)
    hid = torch.empty(3, 16, H, dtype=tdtype(dtype), device="cuda")
    F.fdllm_synth_hidden(11, 3, 4, 64, 16, H, V, 0.5, w, dc, hid)
    ref, planted, _ = synth.hidden_states(11, 3, 4, range(64, 80), H, V, 0.2236, dtype, 0.5)
    assert planted.any() and not planted.all()
    assert np.array_equal(_bits(hid), ref)
    pr = torch.empty(2, 77, dtype=torch.int32, device="cuda")
    F.fdllm_synth_prompt(11, 2, 77, 126464, pr)
    assert np.array_equal(pr.cpu().numpy(), synth.prompt_tokens(11, 2, 77, 126464))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_per_sequence_draws(dtype):
    """Sequence b at its own step and window, and a cache redraw of the flagged sequences only: the
    lock-step draws' bytes for that sequence, step, position and epoch."""
    dc = F.F32 if dtype == "f32" else F.BF16
    steps, starts, epochs = [3, 0, 7], [40, 56, 72], [2, 0, 1]
    i32 = lambda v: torch.tensor(v, dtype=torch.int32, device="cuda")
    q = torch.empty(3, 8, 128, dtype=tdtype(dtype), device="cuda")
    F.fdllm_synth_rows_seq(13, F.SYNTH_KFRESH, 3, i32(steps), i32(starts), 8, 128, 1.0, dc, q)
    for b in range(3):
        ref = synth.per_position(13, synth.KIND_KFRESH, 3, steps[b], range(starts[b], starts[b] + 8), 128, dtype)[b]
        assert np.array_equal(_bits(q)[b], ref)
    V, H = 700, 128
    w = dev(synth.lm_head_weight(13, V, H, 0.2236, dtype), dtype)
    hid = torch.empty(3, 8, H, dtype=tdtype(dtype), device="cuda")
    F.fdllm_synth_hidden_seq(13, 3, i32(steps), i32(starts), 8, H, V, 0.5, w, dc, hid)
    for b in range(3):
        ref, _, _ = synth.hidden_states(13, 3, steps[b], range(starts[b], starts[b] + 8), H, V, 0.2236, dtype, 0.5)
        assert np.array_equal(_bits(hid)[b], ref[b])
    kc = torch.zeros(3, 24, 2, 64, dtype=tdtype(dtype), device="cuda")
    only = torch.tensor([1, 0, 1], dtype=torch.uint8, device="cuda")
    F.fdllm_synth_kv_cache_seq(13, F.SYNTH_VCACHE, 3, 24, 2, 64, i32(epochs), only, 1.0, dc, kc)
    got = _bits(kc)
    for b in range(3):
        ref = synth.kv_cache(13, synth.KIND_VCACHE, 3, 24, 2, 64, epochs[b], dtype)[b]
        assert np.array_equal(got[b], ref) if only[b] else not got[b].any()
