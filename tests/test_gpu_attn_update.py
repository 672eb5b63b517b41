"""fdllm_block_attn_update: the block attention and the cache-window update in one call (the summary's
fused cache update, section 3.4.2 "Cache Overhead and Fused Updates").

Its attention output must equal fdllm_block_attn's bit for bit (the same kernel on the same inputs),
and afterwards the caches must equal the oracle's window splice of the block's fresh K/V bit for bit:
cache rows [s_b, s_b + B) hold the block's keys and values, every other row is unchanged.  Cases cover
DualCache and PrefixCache, lock-step and per-sequence blocks, blocks smaller than / equal to / a
multiple of a key tile, packed KV heads (batch x heads above the SM count), and the shapes the kernel
cannot store itself (the splice kernel then follows the attention, or the call is refused)."""
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


def _bits(t):
    """Stored values as the generator returns them: float32 arrays, or bf16 bit patterns as uint16."""
    if t.dtype == torch.float32:
        return t.cpu().numpy()
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _case(b, P, G, B, k, hq, hkv, d, mode, dtype="bf16", blocks=None, seed=11):
    n = P + G
    desc = F.attn_desc(batch=b, prompt_len=P, gen_length=G, block_size=B, block_idx=k, n_q_heads=hq,
                       n_kv_heads=hkv, head_dim=d, use_cache=1, dual_cache=1 if mode == "dual" else 0,
                       dtype=F.F32 if dtype == "f32" else F.BF16, out_f32=0)
    nq = F.fdllm_attn_query_count(desc)
    kc = synth.kv_cache(seed, synth.KIND_KCACHE, b, n, hkv, d, 0, dtype)
    vc = synth.kv_cache(seed, synth.KIND_VCACHE, b, n, hkv, d, 0, dtype)
    q = synth.kv_cache(seed + 1, synth.KIND_Q, b, nq, hq, d, 0, dtype)
    kf = synth.kv_cache(seed + 2, synth.KIND_KFRESH, b, nq, hkv, d, 0, dtype)
    vf = synth.kv_cache(seed + 3, synth.KIND_VFRESH, b, nq, hkv, d, 0, dtype)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    bi = None if blocks is None else torch.tensor(blocks, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(F.fdllm_attn_workspace_size(desc), 16), dtype=torch.uint8, device="cuda")
    wsb = F.fdllm_attn_workspace_size(desc)
    # reference: the attention alone on copies of the caches
    kc0, vc0 = dev(kc, dtype), dev(vc, dtype)
    out0 = torch.empty(b, nq, hq, d, dtype=tdt, device="cuda")
    if bi is None:
        F.fdllm_block_attn(desc, dev(q, dtype), kc0, vc0, dev(kf, dtype), dev(vf, dtype), out0, None, ws,
                           ws_bytes=wsb)
    else:
        F.fdllm_block_attn_ragged(desc, bi, dev(q, dtype), kc0, vc0, dev(kf, dtype), dev(vf, dtype), out0, None, ws,
                                  ws_bytes=wsb)
    kc1, vc1 = dev(kc, dtype), dev(vc, dtype)
    out1 = torch.empty_like(out0)
    F.fdllm_block_attn_update(desc, bi, dev(q, dtype), kc1, vc1, dev(kf, dtype), dev(vf, dtype), out1, None, ws,
                              ws_bytes=wsb)
    torch.cuda.synchronize()
    assert F.fdllm_last_device_error() == (F.OK, 0)
    assert np.array_equal(_bits(out1), _bits(out0))
    starts = [P + (k if blocks is None else blocks[i]) * B for i in range(b)]
    want_k, want_v = kc.copy(), vc.copy()
    for i in range(b):
        want_k[i:i + 1] = O.kv_splice(kc[i:i + 1], kf[i:i + 1, :B], starts[i])
        want_v[i:i + 1] = O.kv_splice(vc[i:i + 1], vf[i:i + 1, :B], starts[i])
    assert np.array_equal(_bits(kc1), want_k), "k cache"
    assert np.array_equal(_bits(vc1), want_v), "v cache"


@pytest.mark.parametrize("B", [16, 32, 64, 128])
def test_dual_cache_lock_step(B):
    _case(2, 40, 256, B, 1, 4, 4, 128, "dual")


def test_dual_cache_gqa_head_dim_64():
    _case(3, 24, 64, 32, 0, 8, 2, 64, "dual")


def test_prefix_cache_writes_only_the_block():
    _case(2, 40, 128, 32, 1, 4, 4, 128, "prefix")


def test_per_sequence_blocks():
    _case(3, 40, 128, 32, 0, 4, 4, 128, "dual", blocks=[0, 3, 1])


def test_packed_kv_heads():
    # 16 sequences x 32 KV heads: more units than SMs, so KV heads share a 128-row tile (16 keys each)
    _case(16, 64, 64, 32, 1, 32, 32, 128, "dual")


def test_block_not_filling_key_tiles_falls_back_to_the_splice_kernel():
    before = F.fdllm_launch_counter()
    _case(1, 16, 160, 80, 1, 4, 4, 64, "dual")           # 80 rows: a tile and a part of one
    assert F.fdllm_launch_counter() - before == 3        # reference attention; attention + splice


def test_fp32_falls_back_to_the_splice_kernel():
    _case(1, 16, 32, 16, 0, 2, 2, 64, "dual", dtype="f32")


def test_refused_where_the_fallback_cannot_express_the_window():
    desc = F.attn_desc(batch=2, prompt_len=16, gen_length=160, block_size=80, block_idx=0, n_q_heads=4,
                       n_kv_heads=4, head_dim=64, use_cache=1, dual_cache=1, dtype=F.BF16, out_f32=0)
    x = torch.zeros(4096, dtype=torch.bfloat16, device="cuda")
    bi = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(F.FdllmError) as e:
        F.fdllm_block_attn_update(desc, bi, x, x, x, x, x, x)
    assert e.value.status == F.EUNSUPPORTED
    desc.use_cache = 0
    with pytest.raises(F.FdllmError) as e:
        F.fdllm_block_attn_update(desc, None, x, x, x, x, x, x)
    assert e.value.status == F.EUNSUPPORTED


def test_one_launch_per_call():
    before = F.fdllm_launch_counter()
    _case(2, 40, 256, 32, 2, 4, 4, 128, "dual")
    assert F.fdllm_launch_counter() - before == 2        # the reference attention and the fused call
