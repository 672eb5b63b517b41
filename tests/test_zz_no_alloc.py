"""fdllm_confidence_select_noalloc: the confidence select for callers that
cannot allocate device memory (they receive only their input and output
buffers), with the vocabulary partials in the library's fixed device array.

Its outputs must match the workspace entry point's on the same inputs, within
the tolerances of the other parity tests, on two consecutive steps (the second
step sees the tokens the first one unmasked and reuses the array's stale
contents).  This file is collected last so that a run stopping at the first
failure has already run every other test; it also passes alone in a fresh
process."""
import numpy as np
import pytest
import torch

from block_cached_decoding_gb300 import fdllm as F
from block_cached_decoding_gb300 import synth
from gpu_helpers import CONF_ATOL, GAP_EXEMPT, dev, ensure_built, f64, kappa_tol
from oracle import fdllm_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _buffers(b, B):
    return dict(unmasked=torch.zeros(b, B, dtype=torch.uint8, device="cuda"),
                conf=torch.zeros(b, B, dtype=torch.float32, device="cuda"),
                kappa=torch.zeros(b, B, dtype=torch.float32, device="cuda"),
                argmax=torch.zeros(b, B, dtype=torch.int32, device="cuda"),
                n_left=torch.zeros(b, dtype=torch.int32, device="cuda"))


def _host(o):
    return {k: v.cpu().numpy() for k, v in o.items()}


@pytest.mark.parametrize("dtype,batch,B,H,V", [("bf16", 3, 32, 512, 6001),     # tensor-core LM head
                                               ("f32", 2, 16, 256, 1024)])     # CUDA-core LM head
def test_matches_the_workspace_entry_point_on_two_steps(dtype, batch, B, H, V):
    seed, P = 21, 40
    n = P + 2 * B
    s = P
    w = synth.lm_head_weight(seed, V, H, float(np.sqrt(0.02)), dtype)
    w_dev = dev(w, dtype)
    tokens0 = np.full((batch, n), V, dtype=np.int32)
    tokens0[:, :P] = synth.prompt_tokens(seed, batch, P, V)
    t_ref = torch.from_numpy(tokens0.copy()).cuda()
    t_new = torch.from_numpy(tokens0.copy()).cuda()
    desc = F.select_desc(batch=batch, seq_len=n, block_start=s, block_size=B, hidden=H, vocab=V, mask_id=V,
                         threshold=0.9, dtype=F.F32 if dtype == "f32" else F.BF16)
    need = F.fdllm_select_workspace_size(desc)
    assert 0 < need <= F.NOALLOC_SCRATCH_BYTES
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    ref, new = _buffers(batch, B), _buffers(batch, B)
    for step in range(2):
        hid, _, _ = synth.hidden_states(seed, batch, step, range(s, s + B), H, V, float(np.sqrt(0.02)), dtype, 0.4)
        h_dev = dev(hid, dtype)
        F.fdllm_confidence_select(desc, h_dev, w_dev, t_ref, ref["unmasked"], ref["conf"], ref["kappa"],
                                  ref["argmax"], ref["n_left"], ws)
        F.fdllm_confidence_select_noalloc(desc, h_dev, w_dev, t_new, new["unmasked"], new["conf"], new["kappa"],
                                          new["argmax"], new["n_left"])
        torch.cuda.synchronize()
        a, b = _host(ref), _host(new)
        masked = a["argmax"] >= 0
        assert np.array_equal(masked, b["argmax"] >= 0)
        assert np.all(np.isnan(b["conf"][~masked]))
        assert np.abs(a["conf"][masked] - b["conf"][masked]).max(initial=0.0) <= CONF_ATOL
        for x, y in zip(a["kappa"][masked], b["kappa"][masked]):
            assert abs(x - y) <= kappa_tol(x)
        # token ids: equal unless the oracle's top-2 gap is inside the exemption band
        st = O.lm_head_confidence(f64(hid, dtype).reshape(batch * B, H), f64(w, dtype))
        gap = st["gap"].reshape(batch, B)
        diff = (a["argmax"] != b["argmax"]) & masked
        assert np.all(gap[diff] < GAP_EXEMPT)
        if not diff.any():
            assert np.array_equal(a["unmasked"], b["unmasked"])
            assert np.array_equal(t_ref.cpu().numpy(), t_new.cpu().numpy())
            assert np.array_equal(a["n_left"], b["n_left"])
        assert b["unmasked"].sum() >= 1
    assert (t_new.cpu().numpy()[:, s:s + B] != V).sum() >= 2      # both steps unmasked something
    # no device memory is taken by further calls (a stray cudaMalloc inside the library would not
    # show in torch's allocator statistics, but it does in the device's free memory)
    t_new.copy_(torch.from_numpy(tokens0).cuda())
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(5):
        F.fdllm_confidence_select_noalloc(desc, h_dev, w_dev, t_new, new["unmasked"], new["conf"], new["kappa"],
                                          new["argmax"], new["n_left"])
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0


def test_rejects_requests_beyond_the_static_scratch():
    # 2048 block rows: the partials need far more than the 2 MiB array
    desc = F.select_desc(batch=64, seq_len=64, block_start=32, block_size=32, hidden=256, vocab=126464,
                         mask_id=126464, threshold=0.9, dtype=F.BF16)
    assert F.fdllm_select_workspace_size(desc) > F.NOALLOC_SCRATCH_BYTES
    x = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(F.FdllmError) as e:
        F.fdllm_confidence_select_noalloc(desc, x, x, x, x, x, x, x, x)
    assert e.value.status == F.EINVAL and "static scratch" in str(e.value)
