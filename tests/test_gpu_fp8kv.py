"""FP8 KV cache on the GPU: fdllm_kv_splice_fp8 is bit-exact against the oracle's
quantiser (codes and scales), and fdllm_block_attn_fp8kv matches the oracle's block
attention over the dequantised cache (relative L2 <= 5e-3, as for the bf16 cache)."""
import numpy as np
import pytest
import torch

from block_cached_decoding_gb300 import fdllm as F
from block_cached_decoding_gb300 import synth
from gpu_helpers import assert_attention_close, code, dev, ensure_built, f64
from oracle import fdllm_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def fp8_cache(b, n, hkv, d):
    return (torch.zeros(b, n, hkv, d, dtype=torch.uint8, device="cuda"),
            torch.zeros(b, n, hkv, dtype=torch.float32, device="cuda"))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_refresh_then_window_splice_bit_exact(dtype):
    b, n, hkv, d, start, ln = 3, 50, 2, 64, 17, 9
    kc = synth.kv_cache(4, synth.KIND_KCACHE, b, n, hkv, d, 0, dtype)
    vc = synth.kv_cache(4, synth.KIND_VCACHE, b, n, hkv, d, 0, dtype, sigma=30.0)
    ks = synth.kv_cache(5, synth.KIND_KCACHE, b, ln, hkv, d, 0, dtype, sigma=0.01)
    vs = synth.kv_cache(5, synth.KIND_VCACHE, b, ln, hkv, d, 0, dtype)
    kq, ksc = fp8_cache(b, n, hkv, d)
    vq, vsc = fp8_cache(b, n, hkv, d)
    F.fdllm_kv_splice_fp8(F.SPLICE_REFRESH, b, n, hkv, d, 0, n, code(dtype), kq, ksc, vq, vsc, dev(kc, dtype),
                          dev(vc, dtype))
    torch.cuda.synchronize()
    want_kq, want_ks = O.quantize_kv_rows(f64(kc, dtype))
    want_vq, want_vs = O.quantize_kv_rows(f64(vc, dtype))
    assert np.array_equal(kq.cpu().numpy(), want_kq) and np.array_equal(ksc.cpu().numpy(), want_ks)
    assert np.array_equal(vq.cpu().numpy(), want_vq) and np.array_equal(vsc.cpu().numpy(), want_vs)
    F.fdllm_kv_splice_fp8(F.SPLICE_WINDOW, b, n, hkv, d, start, ln, code(dtype), kq, ksc, vq, vsc, dev(ks, dtype),
                          dev(vs, dtype))
    torch.cuda.synchronize()
    want_kq, want_ks = O.kv_splice_fp8(want_kq, want_ks, f64(ks, dtype), start)
    want_vq, want_vs = O.kv_splice_fp8(want_vq, want_vs, f64(vs, dtype), start)
    assert np.array_equal(kq.cpu().numpy(), want_kq) and np.array_equal(ksc.cpu().numpy(), want_ks)
    assert np.array_equal(vq.cpu().numpy(), want_vq) and np.array_equal(vsc.cpu().numpy(), want_vs)


def run_case(*, batch, prompt_len, gen_length, block_size, hq, hkv, d, mode, out_f32=1, block_idx=0, blocks=None,
             seed=7, step=0, poison=False):
    """The cache is drawn in bf16 and written to FP8 by fdllm_kv_splice_fp8 (REFRESH), checked
    against the oracle's codes; the attention is compared with the oracle's over the dequantised
    cache.  `blocks` (a list): sequence b at block blocks[b] (DualCache only).  `poison`: each
    sequence's own window rows of the FP8 cache get NaN codes and NaN scales (rows the attention
    must not use) after the check of the codes."""
    dtype = "bf16"
    n = prompt_len + gen_length
    kc = synth.kv_cache(seed, synth.KIND_KCACHE, batch, n, hkv, d, 0, dtype)
    vc = synth.kv_cache(seed, synth.KIND_VCACHE, batch, n, hkv, d, 0, dtype)
    kq, ksc = fp8_cache(batch, n, hkv, d)
    vq, vsc = fp8_cache(batch, n, hkv, d)
    F.fdllm_kv_splice_fp8(F.SPLICE_REFRESH, batch, n, hkv, d, 0, n, F.BF16, kq, ksc, vq, vsc, dev(kc, dtype),
                          dev(vc, dtype))
    want_kq, want_ks = O.quantize_kv_rows(f64(kc, dtype))
    want_vq, want_vs = O.quantize_kv_rows(f64(vc, dtype))
    torch.cuda.synchronize()
    assert np.array_equal(kq.cpu().numpy(), want_kq) and np.array_equal(vq.cpu().numpy(), want_vq)
    k64, v64 = O.dequantize_kv_rows(want_kq, want_ks), O.dequantize_kv_rows(want_vq, want_vs)
    ks_per = blocks if blocks is not None else [block_idx] * batch
    windows = [O.block_window(prompt_len, block_size, k) for k in ks_per]
    if poison:
        for bi, (s0, e0) in enumerate(windows):
            kq[bi, s0:e0] = 0x7F                           # E4M3 NaN
            vq[bi, s0:e0] = 0xFF
            ksc[bi, s0:e0] = float("nan")
            vsc[bi, s0:e0] = float("inf")
    nq = block_size if mode == "dual" else n - windows[0][0]
    q = np.empty((batch, nq, hq, d), dtype=np.uint16)
    kf = np.empty((batch, nq, hkv, d), dtype=np.uint16)
    vf = np.empty_like(kf)
    for bi, (s, e) in enumerate(windows):
        pos = O.query_positions(mode, s, e, n)
        q[bi] = synth.per_position(seed, synth.KIND_Q, bi + 1, step, pos, hq * d, dtype)[bi].reshape(nq, hq, d)
        kf[bi] = synth.per_position(seed, synth.KIND_KFRESH, bi + 1, step, pos, hkv * d, dtype)[bi].reshape(nq, hkv, d)
        vf[bi] = synth.per_position(seed, synth.KIND_VFRESH, bi + 1, step, pos, hkv * d, dtype)[bi].reshape(nq, hkv, d)
    desc = F.attn_desc(batch=batch, prompt_len=prompt_len, gen_length=gen_length, block_size=block_size,
                       block_idx=block_idx, n_q_heads=hq, n_kv_heads=hkv, head_dim=d, use_cache=1,
                       dual_cache=1 if mode == "dual" else 0, dtype=F.BF16, out_f32=out_f32)
    out = torch.zeros(batch, nq, hq, d, dtype=torch.float32 if out_f32 else torch.bfloat16, device="cuda")
    lse = torch.zeros(batch, nq, hq, dtype=torch.float32, device="cuda")
    wsb = F.fdllm_attn_workspace_size(desc)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda")
    bidx = None if blocks is None else torch.tensor(blocks, dtype=torch.int32, device="cuda")
    assert F.fdllm_last_device_error() == (F.OK, 0)
    F.fdllm_block_attn_fp8kv(desc, bidx, dev(q, dtype), kq, ksc, vq, vsc, dev(kf, dtype), dev(vf, dtype), out, lse,
                             ws, ws_bytes=wsb)
    torch.cuda.synchronize()
    assert F.fdllm_last_device_error() == (F.OK, 0)
    o_gpu = out.float().cpu().numpy().astype(np.float64)
    l_gpu = lse.cpu().numpy()
    worst = 0.0
    for bi, (s, e) in enumerate(windows):
        o_ref, lse_ref = O.block_attention(f64(q[bi:bi + 1], dtype), k64[bi:bi + 1], v64[bi:bi + 1],
                                           f64(kf[bi:bi + 1], dtype), f64(vf[bi:bi + 1], dtype), mode=mode, s=s, e=e,
                                           n_q_heads=hq, n_kv_heads=hkv)
        worst = max(worst, assert_attention_close(o_gpu[bi:bi + 1], o_ref))
        assert np.abs(l_gpu[bi:bi + 1] - lse_ref).max() < 2e-3, bi
    return worst


@pytest.mark.parametrize("mode", ["dual", "prefix"])
@pytest.mark.parametrize("d", [64, 128])
def test_modes(mode, d):
    run_case(batch=2, prompt_len=200, gen_length=96, block_size=32, block_idx=1, hq=4, hkv=4, d=d, mode=mode)


def test_gqa_and_bf16_output():
    run_case(batch=3, prompt_len=45, gen_length=96, block_size=16, block_idx=2, hq=8, hkv=2, d=128, mode="dual",
             out_f32=0)


def test_block_off_the_key_tile():
    run_case(batch=2, prompt_len=77, gen_length=60, block_size=20, block_idx=1, hq=4, hkv=4, d=128, mode="dual")


def test_long_prompt_split_over_the_cluster():
    run_case(batch=1, prompt_len=1500, gen_length=256, block_size=32, block_idx=3, hq=8, hkv=8, d=128, mode="dual")


def test_heads_packed_per_tile():
    """40 sequences x 8 KV heads at block 16: four KV heads share one 128-row query tile."""
    run_case(batch=40, prompt_len=100, gen_length=64, block_size=16, block_idx=2, hq=8, hkv=8, d=64, mode="dual")


def test_each_sequence_at_its_own_block():
    run_case(batch=4, prompt_len=70, gen_length=128, block_size=32, hq=4, hkv=4, d=128, mode="dual",
             blocks=[2, 0, 3, 1])


@pytest.mark.parametrize("d", [64, 128])
def test_window_rows_holding_nan_do_not_reach_the_output(d):
    """NaN codes and NaN / Inf scales in each sequence's own window rows (read with weight zero where a
    key tile crosses the window's edge) leave the output finite and equal to the oracle's."""
    run_case(batch=4, prompt_len=70, gen_length=128, block_size=32, hq=4, hkv=4, d=d, mode="dual",
             blocks=[2, 0, 3, 1], poison=True)


@pytest.mark.parametrize("k", [0, -9, 5, -111, 111])
def test_cache_values_convert_exactly(k):
    """One cache key per head dominates its queries' scores by thousands (its K row is all 256 codes
    with scale 1, the others zero), so the fp32 output is exactly that key's dequantised V row: every
    E4M3 code (normal, subnormal, zero, both signs) times the row's scale 2^k must come out exact,
    for scales from 2^-111 to 2^111 (every value stays a normal float)."""
    b, prompt, gen, B, h, d = 1, 64, 32, 16, 4, 128
    n = prompt + gen
    s = prompt                                           # block 0, DualCache
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F] + [0x01, 0x81], dtype=np.uint8)
    assert len(codes) == 2 * d
    kq = np.zeros((b, n, h, d), dtype=np.uint8)
    vq = np.random.default_rng(3).integers(0, 256, (b, n, h, d)).astype(np.uint8)
    vq[(vq & 0x7F) == 0x7F] = 0x30                       # no NaN codes
    dom = [5, 17, 40, 90]                                # the dominant cache position of each head
    for hh, p in enumerate(dom):
        kq[0, p, hh] = 0x78                              # 256: the score is 2^15
        vq[0, p, hh] = codes[(hh % 2) * d:(hh % 2 + 1) * d]
    # scale 1: the key's raw score q.k is 128 * 256 = 2^15, a power of two, so every product with the
    # softmax scale is exact and the key's weight is exactly 1; every other key's is 2^-4000 = 0
    ksc = np.ones((b, n, h), dtype=np.float32)
    vsc = np.full((b, n, h), 2.0 ** k, dtype=np.float32)
    desc = F.attn_desc(batch=b, prompt_len=prompt, gen_length=gen, block_size=B, block_idx=0, n_q_heads=h,
                       n_kv_heads=h, head_dim=d, use_cache=1, dual_cache=1, dtype=F.BF16, out_f32=1)
    q = torch.ones(b, B, h, d, dtype=torch.bfloat16, device="cuda")
    kf = torch.zeros(b, B, h, d, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(b, B, h, d, dtype=torch.float32, device="cuda")
    ws = torch.empty(max(F.fdllm_attn_workspace_size(desc), 16), dtype=torch.uint8, device="cuda")
    t = lambda x: torch.from_numpy(x).cuda()
    F.fdllm_block_attn_fp8kv(desc, None, q, t(kq), t(ksc), t(vq), t(vsc), kf, kf, out, None, ws,
                             ws_bytes=F.fdllm_attn_workspace_size(desc))
    torch.cuda.synchronize()
    assert F.fdllm_last_device_error() == (F.OK, 0)
    got = out.cpu().numpy()
    for hh, p in enumerate(dom):
        want = (O.e4m3_decode(vq[0, p, hh]) * 2.0 ** k).astype(np.float32)
        for i in range(B):
            assert np.array_equal(got[0, i, hh], want), (hh, i)          # exact values (+0 == -0)


def test_per_sequence_window_splice_bit_exact():
    """Each sequence's window at its own start; an out-of-range start skips its sequence (site 233)."""
    b, n, hkv, d, ln = 4, 60, 2, 128, 12
    starts = [5, 0, 48, 61]                              # the last is out of range
    kc = synth.kv_cache(6, synth.KIND_KCACHE, b, n, hkv, d, 0, "bf16")
    ks = synth.kv_cache(7, synth.KIND_KCACHE, b, ln, hkv, d, 0, "bf16", sigma=3.0)
    vs = synth.kv_cache(7, synth.KIND_VCACHE, b, ln, hkv, d, 0, "bf16")
    want_kq, want_ks = O.quantize_kv_rows(f64(kc, "bf16"))
    kq, ksc = torch.from_numpy(want_kq).cuda(), torch.from_numpy(want_ks.astype(np.float32)).cuda()
    vq, vsc = kq.clone(), ksc.clone()
    assert F.fdllm_last_device_error() == (F.OK, 0)
    F.fdllm_kv_splice_fp8_ragged(b, n, hkv, d, torch.tensor(starts, dtype=torch.int32, device="cuda"), ln, F.BF16,
                                 kq, ksc, vq, vsc, dev(ks, "bf16"), dev(vs, "bf16"))
    assert F.fdllm_last_device_error() == (F.EINVAL, 233)
    got_kq, got_ks, got_vq = kq.cpu().numpy(), ksc.cpu().numpy(), vq.cpu().numpy()
    for i, s in enumerate(starts):
        if s + ln <= n:
            wk, wks = O.kv_splice_fp8(want_kq[i:i + 1], want_ks[i:i + 1], f64(ks[i:i + 1], "bf16"), s)
            wv, _ = O.kv_splice_fp8(want_kq[i:i + 1], want_ks[i:i + 1], f64(vs[i:i + 1], "bf16"), s)
        else:
            wk, wks, wv = want_kq[i:i + 1], want_ks[i:i + 1], want_kq[i:i + 1]
        assert np.array_equal(got_kq[i:i + 1], wk) and np.array_equal(got_ks[i:i + 1], wks)
        assert np.array_equal(got_vq[i:i + 1], wv)


def _random_fp8_cache(rng, b, n, hkv, d):
    """Seeded E4M3 codes drawn directly (random sign, exponent field 4..10, any mantissa: magnitudes
    1/8..15) with power-of-two row scales 2^-3..2^0: a cache of a benchmark shape without running a
    quantiser over it."""
    raw = np.frombuffer(rng.bytes(b * n * hkv * d), dtype=np.uint8).reshape(b, n, hkv, d)
    codes = (raw & 0x87) | ((((raw >> 3) & 0xF) % 7 + 4) << 3)   # sign and mantissa kept, exponent 4..10
    scales = np.exp2(rng.integers(-3, 1, size=(b, n, hkv))).astype(np.float32)
    return codes, scales


def _bf16_normals(rng, shape):
    return torch.from_numpy(rng.standard_normal(shape, dtype=np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("shape", [dict(batch=16, prompt_len=768, gen_length=256, hq=32, hkv=32),
                                   dict(batch=8, prompt_len=512, gen_length=1024, hq=28, hkv=4)],
                         ids=["llada-dual-batch16", "dream-gqa-batch8"])
def test_benchmark_shapes_sampled_sequences(shape):
    """The benchmark's FP8-cache launch configurations: LLaDA DualCache at batch 16 (four KV heads per
    tile, 64 key tiles per CTA, so the ring wraps many times over tiles of both softmax groups) and Dream
    GQA at batch 8.  Every query row of two sampled sequences against the oracle's attention over the
    dequantised cache."""
    b, prompt_len, gen_length, hq, hkv = (shape[k] for k in ("batch", "prompt_len", "gen_length", "hq", "hkv"))
    d, block_size, block_idx = 128, 32, 0
    n = prompt_len + gen_length
    rng = np.random.default_rng(11 + b)
    kq, ks = _random_fp8_cache(rng, b, n, hkv, d)
    vq, vs = _random_fp8_cache(rng, b, n, hkv, d)
    q = _bf16_normals(rng, (b, block_size, hq, d))
    kf = _bf16_normals(rng, (b, block_size, hkv, d))
    vf = _bf16_normals(rng, (b, block_size, hkv, d))
    desc = F.attn_desc(batch=b, prompt_len=prompt_len, gen_length=gen_length, block_size=block_size,
                       block_idx=block_idx, n_q_heads=hq, n_kv_heads=hkv, head_dim=d, use_cache=1, dual_cache=1,
                       dtype=F.BF16, out_f32=1)
    assert F.fdllm_attn_query_count(desc) == block_size
    out = torch.zeros(b, block_size, hq, d, dtype=torch.float32, device="cuda")
    lse = torch.zeros(b, block_size, hq, dtype=torch.float32, device="cuda")
    wsb = F.fdllm_attn_workspace_size(desc)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda")
    t = lambda x: torch.from_numpy(x).cuda()
    assert F.fdllm_last_device_error() == (F.OK, 0)
    F.fdllm_block_attn_fp8kv(desc, None, q.cuda(), t(kq), t(ks), t(vq), t(vs), kf.cuda(), vf.cuda(), out, lse, ws,
                             ws_bytes=wsb)
    torch.cuda.synchronize()
    assert F.fdllm_last_device_error() == (F.OK, 0)
    o_gpu = out.cpu().numpy().astype(np.float64)
    l_gpu = lse.cpu().numpy()
    s, e = O.block_window(prompt_len, block_size, block_idx)
    f = lambda x: x.float().numpy().astype(np.float64)
    for bi in sorted(rng.choice(b, size=2, replace=False).tolist()):
        sl = slice(bi, bi + 1)
        o_ref, lse_ref = O.block_attention(f(q[sl]), O.dequantize_kv_rows(kq[sl], ks[sl]),
                                           O.dequantize_kv_rows(vq[sl], vs[sl]), f(kf[sl]), f(vf[sl]), mode="dual",
                                           s=s, e=e, n_q_heads=hq, n_kv_heads=hkv)
        assert_attention_close(o_gpu[sl], o_ref)
        assert np.abs(l_gpu[sl] - lse_ref).max() < 2e-3, bi
