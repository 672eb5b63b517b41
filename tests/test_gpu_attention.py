"""fdllm_block_attn against the oracle's block attention (relative L2 <= 5e-3)."""
import numpy as np
import pytest
import torch

from block_cached_decoding_gb300 import configs
from block_cached_decoding_gb300 import fdllm as F
from block_cached_decoding_gb300 import synth
from gpu_helpers import assert_attention_close, code, dev, ensure_built, f64, tdtype
from oracle import fdllm_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def run_case(*, batch, prompt_len, gen_length, block_size, block_idx, hq, hkv, d, mode, dtype, seed=0, step=0,
             out_f32=1):
    n = prompt_len + gen_length
    s, e = O.block_window(prompt_len, block_size, block_idx)
    pos = O.query_positions(mode, s, e, n)
    kc = synth.kv_cache(seed, synth.KIND_KCACHE, batch, n, hkv, d, block_idx, dtype)
    vc = synth.kv_cache(seed, synth.KIND_VCACHE, batch, n, hkv, d, block_idx, dtype)
    q = synth.per_position(seed, synth.KIND_Q, batch, step, pos, hq * d, dtype).reshape(batch, len(pos), hq, d)
    kf = synth.per_position(seed, synth.KIND_KFRESH, batch, step, pos, hkv * d, dtype).reshape(batch, len(pos), hkv, d)
    vf = synth.per_position(seed, synth.KIND_VFRESH, batch, step, pos, hkv * d, dtype).reshape(batch, len(pos), hkv, d)
    o_ref, lse_ref = O.block_attention(f64(q, dtype), f64(kc, dtype), f64(vc, dtype), f64(kf, dtype), f64(vf, dtype),
                                       mode=mode, s=s, e=e, n_q_heads=hq, n_kv_heads=hkv)
    desc = F.attn_desc(batch=batch, prompt_len=prompt_len, gen_length=gen_length, block_size=block_size,
                       block_idx=block_idx, n_q_heads=hq, n_kv_heads=hkv, head_dim=d,
                       use_cache=0 if mode == "none" else 1, dual_cache=1 if mode == "dual" else 0,
                       dtype=code(dtype), out_f32=out_f32)
    assert F.fdllm_attn_query_count(desc) == len(pos)
    out = torch.empty(batch, len(pos), hq, d, dtype=torch.float32 if out_f32 else tdtype(dtype), device="cuda")
    lse = torch.empty(batch, len(pos), hq, dtype=torch.float32, device="cuda")
    wsb = F.fdllm_attn_workspace_size(desc)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda")
    F.fdllm_block_attn(desc, dev(q, dtype), dev(kc, dtype), dev(vc, dtype), dev(kf, dtype), dev(vf, dtype), out,
                       lse, ws, ws_bytes=wsb)
    torch.cuda.synchronize()
    worst = assert_attention_close(out.float().cpu().numpy().astype(np.float64), o_ref)
    assert np.abs(lse.cpu().numpy() - lse_ref).max() < 2e-3
    return worst


def test_tiny_fp32_every_block():
    wl = configs.TINY
    for k in range(wl.gen_length // wl.block_size):
        run_case(batch=1, prompt_len=wl.prompt_len, gen_length=wl.gen_length, block_size=wl.block_size,
                 block_idx=k, hq=wl.n_q_heads, hkv=wl.n_kv_heads, d=wl.head_dim, mode="dual", dtype="f32",
                 seed=wl.seed, step=k)


@pytest.mark.parametrize("mode", ["dual", "prefix", "none"])
@pytest.mark.parametrize("d", [64, 128])
def test_bf16_modes(mode, d):
    run_case(batch=2, prompt_len=200, gen_length=96, block_size=32, block_idx=1, hq=4, hkv=4, d=d, mode=mode,
             dtype="bf16", seed=3)


@pytest.mark.parametrize("batch,hq,d,block,prompt,gen,out_f32", [
    (40, 8, 64, 16, 100, 64, 0),     # 320 head units > 152 SMs: 4 KV heads per tile, bf16 output
    (24, 8, 128, 32, 90, 96, 1),     # 192 units: 2 per tile
    (30, 6, 128, 20, 77, 60, 0),     # 6 heads: 2 per tile; ragged block and key counts
    (48, 4, 64, 64, 40, 128, 1)])    # 64 queries: 2 per tile at most
def test_mha_heads_packed_per_tile(batch, hq, d, block, prompt, gen, out_f32):
    """MHA with a block of at most 64 queries and more (sequence, head) units than one wave of
    CTAs packs 2 or 4 KV heads into one 128-row tile: row r's head owns a block of each score tile
    and of P (the rest of the row is zero)."""
    run_case(batch=batch, prompt_len=prompt, gen_length=gen, block_size=block, block_idx=1, hq=hq, hkv=hq, d=d,
             mode="dual", dtype="bf16", seed=9, out_f32=out_f32)


@pytest.mark.parametrize("prompt,gen,block,k,hq,hkv,d", [
    (100, 64, 16, 0, 4, 4, 128),     # 16 fresh rows + the suffix's last 48: one full joined tile
    (100, 32, 16, 0, 4, 4, 64),      # 16 fresh + 16 suffix rows; the rest of the joined tile past the cache
    (64, 128, 8, 1, 8, 2, 128),      # 8 fresh + 48 suffix rows, grouped-query heads
    (40, 192, 48, 1, 4, 4, 128),     # 48 fresh + 32 suffix rows do not fit one tile: no joined tile
    (200, 96, 32, 1, 28, 4, 128)])   # the Dream head layout, 32 + 32 rows
def test_dual_fresh_tile_joined_with_suffix_tail(prompt, gen, block, k, hq, hkv, d):
    """DualCache with fewer fresh rows than a key tile: when the suffix's last, partial tile fits
    beside them, both share one tile (the fresh rows, then the cached tail), so the unit has one key
    tile less; the attention over every position must not change."""
    run_case(batch=3, prompt_len=prompt, gen_length=gen, block_size=block, block_idx=k, hq=hq, hkv=hkv, d=d,
             mode="dual", dtype="bf16", seed=12, out_f32=0)


@pytest.mark.parametrize("hq,hkv", [(28, 4), (8, 1), (6, 2)])
def test_bf16_gqa(hq, hkv):
    run_case(batch=2, prompt_len=130, gen_length=64, block_size=32, block_idx=0, hq=hq, hkv=hkv, d=128,
             mode="dual", dtype="bf16", seed=4)


@pytest.mark.parametrize("case", [
    dict(batch=1, prompt_len=0, gen_length=16, block_size=16, block_idx=0),    # no prompt, one block
    dict(batch=3, prompt_len=37, gen_length=60, block_size=20, block_idx=2),   # ragged block, last block
    dict(batch=1, prompt_len=5, gen_length=3, block_size=1, block_idx=1),      # block of one
    dict(batch=1, prompt_len=300, gen_length=257 * 4, block_size=257, block_idx=3),
    dict(batch=2, prompt_len=3000, gen_length=128, block_size=32, block_idx=1)])   # > 16 key tiles: fp32 partials
def test_bf16_ragged(case):
    run_case(hq=4, hkv=2, d=128, mode="dual", dtype="bf16", seed=5, **case)


def test_bf16_output_in_input_dtype():
    run_case(batch=1, prompt_len=64, gen_length=64, block_size=32, block_idx=1, hq=4, hkv=4, d=128, mode="dual",
             dtype="bf16", seed=6, out_f32=0)
