"""fdllm_kv_splice is bit-exact against the oracle's splice (window and refresh)."""
import numpy as np
import pytest
import torch

from block_cached_decoding_gb300 import fdllm as F
from block_cached_decoding_gb300 import synth
from gpu_helpers import dev, ensure_built
from oracle import fdllm_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


@pytest.mark.parametrize("dtype,b,n,hkv,d,start,ln", [
    ("bf16", 2, 96, 4, 64, 40, 16), ("f32", 1, 128, 4, 64, 64, 16), ("bf16", 3, 50, 1, 128, 49, 1),
    ("bf16", 2, 96, 4, 64, 0, 96), ("bf16", 1, 64, 2, 64, 10, 0)])
def test_window(dtype, b, n, hkv, d, start, ln):
    kc = synth.kv_cache(1, synth.KIND_KCACHE, b, n, hkv, d, 0, dtype)
    vc = synth.kv_cache(1, synth.KIND_VCACHE, b, n, hkv, d, 0, dtype)
    ks = synth.kv_cache(2, synth.KIND_KCACHE, b, ln, hkv, d, 0, dtype) if ln else kc[:, :0]
    vs = synth.kv_cache(2, synth.KIND_VCACHE, b, ln, hkv, d, 0, dtype) if ln else vc[:, :0]
    tk, tv = dev(kc, dtype), dev(vc, dtype)
    sk, sv = (dev(ks, dtype), dev(vs, dtype)) if ln else (tk, tv)
    mode = F.SPLICE_REFRESH if (start == 0 and ln == n) else F.SPLICE_WINDOW
    F.fdllm_kv_splice(mode, b, n, hkv, d, start, ln, F.F32 if dtype == "f32" else F.BF16, tk, tv, sk, sv)
    torch.cuda.synchronize()
    view = (lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)) if dtype == "bf16" else (lambda t: t.cpu().numpy())
    assert np.array_equal(view(tk), O.kv_splice(kc, ks, start))
    assert np.array_equal(view(tv), O.kv_splice(vc, vs, start))
