"""Host-side guards of the C ABI that need a GPU to exercise: the clustered LM head
(more than 128 block rows: operand tiles multicast between the CTAs of a
thread-block cluster) accepts only device memory of the current device, and
rejects host memory with FDLLM_EINVAL before anything is launched."""
import numpy as np
import pytest
import torch

from block_cached_decoding_gb300 import fdllm as F
from block_cached_decoding_gb300 import synth
from gpu_helpers import SelectOutputs, dev, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _problem(batch, B=32, H=256, V=3001, seed=5):
    P = 16
    n = P + B
    w = synth.lm_head_weight(seed, V, H, float(np.sqrt(0.02)), "bf16")
    hid, _, _ = synth.hidden_states(seed, batch, 0, range(P, P + B), H, V, float(np.sqrt(0.02)), "bf16", 0.4)
    tokens = np.full((batch, n), V, dtype=np.int32)
    tokens[:, :P] = 3
    desc = F.select_desc(batch=batch, seq_len=n, block_start=P, block_size=B, hidden=H, vocab=V, mask_id=V,
                         threshold=0.9, dtype=F.BF16)
    return desc, dev(hid, "bf16"), dev(w, "bf16"), torch.from_numpy(tokens).cuda()


@pytest.mark.parametrize("which", ["hidden", "lm_head_w"])
def test_clustered_lm_head_rejects_host_memory(which):
    desc, h, w, t = _problem(batch=8)                 # 256 block rows: clusters of 2 CTAs
    outs = SelectOutputs(desc, 8, 32)
    host = (h if which == "hidden" else w).cpu().pin_memory()
    args = (host, w) if which == "hidden" else (h, host)
    before = t.clone()
    with pytest.raises(F.FdllmError) as e:
        F.fdllm_confidence_select(desc, *args, t, outs.unmasked, outs.conf, outs.kappa, outs.argmax, outs.n_left,
                                  outs.ws)
    assert e.value.status == F.EINVAL and which in str(e.value)
    torch.cuda.synchronize()
    assert torch.equal(t, before)                      # nothing ran
    with pytest.raises(F.FdllmError) as e:
        F.fdllm_confidence_select_noalloc(desc, *args, t, outs.unmasked, outs.conf, outs.kappa, outs.argmax,
                                          outs.n_left)
    assert e.value.status == F.EINVAL
    assert F.fdllm_last_device_error() == (F.OK, 0)


def test_clustered_lm_head_accepts_device_memory():
    desc, h, w, t = _problem(batch=8)
    outs = SelectOutputs(desc, 8, 32)
    outs.run(desc, h, w, t)
    got = outs.host()
    assert np.all(got["unmask"].sum(axis=1) >= 1)
    assert F.fdllm_last_device_error() == (F.OK, 0)
