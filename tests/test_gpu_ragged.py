"""Per-sequence (non-lock-step) blocks: each sequence of the batch sits at its own
block.  Every call is compared with the oracle run on that sequence alone at its
own block window; a short generation in which each sequence moves to its next
block as soon as its own block is decoded is checked step by step."""
import numpy as np
import pytest
import torch

from block_cached_decoding_gb300 import fdllm as F
from block_cached_decoding_gb300 import synth
from gpu_helpers import SelectOutputs, assert_attention_close, code, compare_select, dev, ensure_built, f64
from oracle import fdllm_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _ints(a):
    return torch.tensor(np.asarray(a, dtype=np.int32), device="cuda")


def seq_rows(seed, kind, b, step, positions, width, dtype):
    return synth.per_position(seed, kind, b + 1, step, positions, width, dtype)[b]


def seq_hidden(seed, b, step, positions, H, V, sigma, dtype, p_plant):
    return synth.hidden_states(seed, b + 1, step, positions, H, V, sigma, dtype, p_plant)[0][b]


def seq_cache(seed, kind, b, n, hkv, d, epoch, dtype):
    return synth.kv_cache(seed, kind, b + 1, n, hkv, d, epoch, dtype)[b]


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------

def ragged_attention_case(*, blocks, prompt_len, gen_length, block_size, hq, hkv, d, out_f32, seed=3, step=0,
                          bad=None, poison=False):
    """Sequence b at block blocks[b]; returns the worst relative L2 over valid sequences.

    `bad` (a sequence index) has its block index replaced by an out-of-range one.  `poison` writes NaN
    and Inf into each sequence's own window rows of the cache (rows the attention must not use)."""
    batch = len(blocks)
    n = prompt_len + gen_length
    dtype = "bf16"
    kc = synth.kv_cache(seed, synth.KIND_KCACHE, batch, n, hkv, d, 0, dtype)
    vc = synth.kv_cache(seed, synth.KIND_VCACHE, batch, n, hkv, d, 0, dtype)
    q = np.empty((batch, block_size, hq, d), dtype=np.uint16)
    kf = np.empty((batch, block_size, hkv, d), dtype=np.uint16)
    vf = np.empty_like(kf)
    for b, k in enumerate(blocks):
        s, e = O.block_window(prompt_len, block_size, k)
        q[b] = seq_rows(seed, synth.KIND_Q, b, step, range(s, e), hq * d, dtype).reshape(block_size, hq, d)
        kf[b] = seq_rows(seed, synth.KIND_KFRESH, b, step, range(s, e), hkv * d, dtype).reshape(block_size, hkv, d)
        vf[b] = seq_rows(seed, synth.KIND_VFRESH, b, step, range(s, e), hkv * d, dtype).reshape(block_size, hkv, d)
    idx = list(blocks)
    if bad is not None:
        idx[bad] = gen_length // block_size
    kc_in, vc_in = kc, vc
    if poison:
        kc_in, vc_in = kc.copy(), vc.copy()
        for b, k in enumerate(blocks):
            s, e = O.block_window(prompt_len, block_size, k)
            kc_in[b, s:e] = 0x7FC0                       # bf16 NaN
            vc_in[b, s:e] = 0x7F80                       # bf16 +Inf
    desc = F.attn_desc(batch=batch, prompt_len=prompt_len, gen_length=gen_length, block_size=block_size,
                       block_idx=0, n_q_heads=hq, n_kv_heads=hkv, head_dim=d, use_cache=1, dual_cache=1,
                       dtype=F.BF16, out_f32=out_f32)
    out = torch.full((batch, block_size, hq, d), 0.0, dtype=torch.float32 if out_f32 else torch.bfloat16,
                     device="cuda")
    lse = torch.zeros(batch, block_size, hq, dtype=torch.float32, device="cuda")
    wsb = F.fdllm_attn_workspace_size(desc)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda")
    assert F.fdllm_last_device_error() == (F.OK, 0)
    F.fdllm_block_attn_ragged(desc, _ints(idx), dev(q, dtype), dev(kc_in, dtype), dev(vc_in, dtype), dev(kf, dtype),
                              dev(vf, dtype), out, lse, ws, ws_bytes=wsb)
    torch.cuda.synchronize()
    err = F.fdllm_last_device_error()
    assert err == ((F.EINVAL, 232) if bad is not None else (F.OK, 0))
    o_gpu = out.float().cpu().numpy().astype(np.float64)
    l_gpu = lse.cpu().numpy()
    worst = 0.0
    for b, k in enumerate(blocks):
        if b == bad:
            continue
        s, e = O.block_window(prompt_len, block_size, k)
        o_ref, lse_ref = O.block_attention(f64(q[b:b + 1], dtype), f64(kc[b:b + 1], dtype), f64(vc[b:b + 1], dtype),
                                           f64(kf[b:b + 1], dtype), f64(vf[b:b + 1], dtype), mode="dual", s=s, e=e,
                                           n_q_heads=hq, n_kv_heads=hkv)
        worst = max(worst, assert_attention_close(o_gpu[b:b + 1], o_ref))
        assert np.abs(l_gpu[b:b + 1] - lse_ref).max() < 2e-3, b
    return worst


@pytest.mark.parametrize("blocks,prompt,gen,B,hq,hkv,d,out_f32", [
    ([2, 0, 3, 1], 70, 128, 32, 4, 4, 128, 1),        # every block once, MHA
    ([5, 0, 2], 45, 96, 16, 8, 2, 64, 0),             # GQA, bf16 output
    ([2, 0, 1], 77, 60, 20, 4, 4, 128, 1),            # block size off the key tile: ragged tile edges
    ([7, 1], 1500, 256, 32, 8, 8, 128, 1),            # long prompt: split KV merged across the cluster
    ([0], 64, 64, 64, 2, 1, 64, 0),                   # one sequence, block = one key tile
])
def test_attention_each_sequence_at_its_own_block(blocks, prompt, gen, B, hq, hkv, d, out_f32):
    ragged_attention_case(blocks=blocks, prompt_len=prompt, gen_length=gen, block_size=B, hq=hq, hkv=hkv, d=d,
                          out_f32=out_f32)


@pytest.mark.parametrize("blocks,prompt,gen,B,hq,hkv,d", [
    ([2, 0, 3, 1], 70, 128, 32, 4, 4, 128),           # windows off the 64-key tile boundaries
    ([1, 2], 77, 60, 20, 4, 4, 64),                   # block size off the key tile
])
def test_window_rows_holding_nan_and_inf_do_not_reach_the_output(blocks, prompt, gen, B, hq, hkv, d):
    """A key tile at the edge of the prefix reads cache rows of the sequence's own window with weight
    zero; NaN keys and infinite values there must leave the output finite and equal to the oracle's
    (which never reads those rows)."""
    ragged_attention_case(blocks=blocks, prompt_len=prompt, gen_length=gen, block_size=B, hq=hq, hkv=hkv, d=d,
                          out_f32=1, poison=True)


def test_attention_heads_packed_per_tile():
    """40 sequences x 8 KV heads at block 16: four KV heads share one 128-row query tile."""
    rng = np.random.default_rng(11)
    blocks = rng.integers(0, 4, 40).tolist()
    ragged_attention_case(blocks=blocks, prompt_len=100, gen_length=64, block_size=16, hq=8, hkv=8, d=64,
                          out_f32=1)


@pytest.mark.parametrize("bad", [0, 2])
def test_attention_out_of_range_block_is_reported(bad):
    """A block index outside [0, gen / B) skips that sequence and reports EINVAL (site 232);
    the other sequences are still exact."""
    ragged_attention_case(blocks=[1, 3, 0], prompt_len=50, gen_length=128, block_size=32, hq=4, hkv=4, d=128,
                          out_f32=1, bad=bad)


# ---------------------------------------------------------------------------
# confidence select
# ---------------------------------------------------------------------------

_W = {}


def weight(seed, V, H, sigma, dtype):
    key = (seed, V, H, sigma, dtype)
    if key not in _W:
        w = synth.lm_head_weight(seed, V, H, sigma, dtype)
        _W[key] = (dev(w, dtype), f64(w, dtype))
    return _W[key]


def ragged_select_case(*, blocks, prompt_len, gen_length, B, H, V, dtype, tau=0.9, p_plant=0.4, seed=5, step=0,
                       decoded=0.0, bad=None):
    batch = len(blocks)
    n = prompt_len + gen_length
    sigma = float(np.sqrt(0.02))
    w_dev, w64 = weight(seed, V, H, sigma, dtype)
    rng = np.random.default_rng(seed * 131 + batch)
    tokens = np.full((batch, n), V, dtype=np.int64)
    tokens[:, :prompt_len] = synth.prompt_tokens(seed, batch, prompt_len, V)
    starts = [O.block_window(prompt_len, B, k)[0] for k in blocks]
    hid = np.empty((batch, B, H), dtype=np.float32 if dtype == "f32" else np.uint16)
    for b, s in enumerate(starts):
        tokens[b, :s] = np.where(tokens[b, :s] == V, 7, tokens[b, :s])       # earlier blocks decoded
        tokens[b, s:s + B] = np.where(rng.random(B) < decoded, 5, V)         # part of this block decoded
        hid[b] = seq_hidden(seed, b, step, range(s, s + B), H, V, sigma, dtype, p_plant)
    # the oracle on each sequence alone, at its own window
    info = {}
    ref_tokens = tokens.copy()
    for b, s in enumerate(starts):
        t_b, i_b = O.decode_step(tokens[b:b + 1], f64(hid[b:b + 1], dtype), w64, s=s, block_size=B, mask_id=V,
                                 tau=tau)
        ref_tokens[b] = t_b[0]
        for key, val in i_b.items():
            info.setdefault(key, []).append(val)
    info = {k: np.concatenate(v) for k, v in info.items()}
    dev_starts = list(starts)
    if bad is not None:
        dev_starts[bad] = n - B + 1
    desc = F.select_desc(batch=batch, seq_len=n, block_start=prompt_len, block_size=B, hidden=H, vocab=V,
                         mask_id=V, threshold=tau, dtype=code(dtype))
    t_dev = torch.from_numpy(tokens.astype(np.int32)).cuda()
    outs = SelectOutputs(desc, batch, B)
    assert F.fdllm_last_device_error() == (F.OK, 0)
    F.fdllm_confidence_select_ragged(desc, _ints(dev_starts), dev(hid, dtype), w_dev, t_dev, outs.unmasked, outs.conf,
                                     outs.kappa, outs.argmax, outs.n_left, outs.ws)
    got = outs.host()
    err = F.fdllm_last_device_error()
    assert err == ((F.EINVAL, 231) if bad is not None else (F.OK, 0))
    t_got = t_dev.cpu().numpy()
    if bad is not None:
        # the skipped sequence: nothing read, nothing written, reported as nothing masked
        assert np.array_equal(t_got[bad], tokens[bad])
        assert not got["unmask"][bad].any() and got["n_left"][bad] == 0
        keep = [b for b in range(batch) if b != bad]
        info = {k: v[keep] for k, v in info.items()}
        got = {k: v[keep] for k, v in got.items()}
        t_got, tokens, starts = t_got[keep], tokens[keep], [starts[b] for b in keep]
    compare_select(info, got, tau)
    for b, s in enumerate(starts):
        changed = np.nonzero(t_got[b] != tokens[b])[0]
        assert np.all((changed >= s) & (changed < s + B)), (b, changed)
        for i in np.nonzero(got["unmask"][b])[0]:
            assert t_got[b, s + i] == got["token"][b, i]
        assert got["n_left"][b] == (t_got[b, s:s + B] == V).sum()
    return info, got


@pytest.mark.parametrize("blocks,B,H,V,dtype,decoded", [
    ([3, 0, 1, 3, 2], 32, 256, 5000, "bf16", 0.0),     # tensor-core LM head, one row tile
    ([1, 0, 2], 16, 128, 1000, "f32", 0.3),            # fp32 path, partly decoded blocks
    ([0, 3, 2, 1, 0, 3, 1, 2], 32, 192, 3000, "bf16", 0.5),   # 256 block rows: two row tiles
])
def test_select_each_sequence_at_its_own_block(blocks, B, H, V, dtype, decoded):
    ragged_select_case(blocks=blocks, prompt_len=40, gen_length=4 * B, B=B, H=H, V=V, dtype=dtype, decoded=decoded)


def test_select_many_sequences_per_selector():
    rng = np.random.default_rng(2)
    blocks = rng.integers(0, 8, 32).tolist()
    ragged_select_case(blocks=blocks, prompt_len=21, gen_length=32, B=4, H=128, V=200, dtype="bf16", p_plant=0.6)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_select_out_of_range_start_is_reported(dtype):
    ragged_select_case(blocks=[1, 0, 2], prompt_len=30, gen_length=64, B=16, H=128, V=700, dtype=dtype, bad=1)


# ---------------------------------------------------------------------------
# window splice
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,n,hkv,d,starts,ln", [
    ("bf16", 96, 4, 64, [10, 0, 80], 16),
    ("f32", 64, 2, 64, [48, 5], 16),
    ("bf16", 50, 1, 128, [49, 0, 7, 33], 1),
])
def test_splice_each_sequence_at_its_own_window(dtype, n, hkv, d, starts, ln):
    b = len(starts)
    kc = synth.kv_cache(1, synth.KIND_KCACHE, b, n, hkv, d, 0, dtype)
    vc = synth.kv_cache(1, synth.KIND_VCACHE, b, n, hkv, d, 0, dtype)
    ks = synth.kv_cache(2, synth.KIND_KCACHE, b, ln, hkv, d, 0, dtype)
    vs = synth.kv_cache(2, synth.KIND_VCACHE, b, ln, hkv, d, 0, dtype)
    tk, tv = dev(kc, dtype), dev(vc, dtype)
    F.fdllm_kv_splice_ragged(b, n, hkv, d, _ints(starts), ln, code(dtype), tk, tv, dev(ks, dtype), dev(vs, dtype))
    torch.cuda.synchronize()
    view = (lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)) if dtype == "bf16" else (lambda t: t.cpu().numpy())
    gk, gv = view(tk), view(tv)
    for i, s in enumerate(starts):
        assert np.array_equal(gk[i:i + 1], O.kv_splice(kc[i:i + 1], ks[i:i + 1], s))
        assert np.array_equal(gv[i:i + 1], O.kv_splice(vc[i:i + 1], vs[i:i + 1], s))


@pytest.mark.parametrize("bad_start", [-1, 81])
def test_splice_out_of_range_window_is_reported(bad_start):
    n, hkv, d, ln = 96, 2, 64, 16
    kc = synth.kv_cache(1, synth.KIND_KCACHE, 2, n, hkv, d, 0, "bf16")
    ks = synth.kv_cache(2, synth.KIND_KCACHE, 2, ln, hkv, d, 0, "bf16")
    tk, tv = dev(kc, "bf16"), dev(kc, "bf16")
    assert F.fdllm_last_device_error() == (F.OK, 0)
    F.fdllm_kv_splice_ragged(2, n, hkv, d, _ints([30, bad_start]), ln, F.BF16, tk, tv, dev(ks, "bf16"),
                             dev(ks, "bf16"))
    assert F.fdllm_last_device_error() == (F.EINVAL, 233)
    gk = tk.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(gk[:1], O.kv_splice(kc[:1], ks[:1], 30))
    assert np.array_equal(gk[1], kc[1])                  # the skipped sequence is untouched


# ---------------------------------------------------------------------------
# a short generation, each sequence at its own pace
# ---------------------------------------------------------------------------

def test_generation_with_sequences_at_their_own_blocks():
    """Each sequence advances to its next block as soon as its own block is decoded
    (its cache is then refreshed for that block and its fresh window spliced in);
    every step is checked against the oracle on the GPU's current state."""
    seed, batch, prompt_len, B, nblk = 9, 4, 40, 16, 4
    hq, hkv, d, H, V, tau, p_plant = 4, 2, 128, 256, 1500, 0.9, 0.3
    n = prompt_len + nblk * B
    sigma = float(np.sqrt(0.02))
    dtype = "bf16"
    w_dev, w64 = weight(seed, V, H, sigma, dtype)
    tokens0 = np.full((batch, n), V, dtype=np.int64)
    tokens0[:, :prompt_len] = synth.prompt_tokens(seed, batch, prompt_len, V)
    t_dev = torch.from_numpy(tokens0.astype(np.int32)).cuda()
    blk = [0] * batch          # each sequence's block
    step = [0] * batch         # each sequence's own step counter
    # caches: sequence b holds the draw of refresh epoch blk[b]
    kc = np.stack([seq_cache(seed, synth.KIND_KCACHE, b, n, hkv, d, 0, dtype) for b in range(batch)])
    vc = np.stack([seq_cache(seed, synth.KIND_VCACHE, b, n, hkv, d, 0, dtype) for b in range(batch)])
    kc_dev, vc_dev = dev(kc, dtype), dev(vc, dtype)
    adesc = F.attn_desc(batch=batch, prompt_len=prompt_len, gen_length=nblk * B, block_size=B, block_idx=0,
                        n_q_heads=hq, n_kv_heads=hkv, head_dim=d, use_cache=1, dual_cache=1, dtype=F.BF16, out_f32=1)
    sdesc = F.select_desc(batch=batch, seq_len=n, block_start=prompt_len, block_size=B, hidden=H, vocab=V,
                          mask_id=V, threshold=tau, dtype=F.BF16)
    wsb = F.fdllm_attn_workspace_size(adesc)
    aws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda")
    outs = SelectOutputs(sdesc, batch, B)
    out = torch.empty(batch, B, hq, d, dtype=torch.float32, device="cuda")
    done = [False] * batch
    steps_in_block = [0] * batch
    advanced = 0
    exempt = 0
    apart = 0                  # steps at which the sequences were not all at the same block
    for it in range(nblk * B + 1):
        if all(done):
            break
        starts = [prompt_len + k * B for k in blk]
        apart += len(set(blk)) > 1
        q = np.stack([seq_rows(seed, synth.KIND_Q, b, step[b], range(starts[b], starts[b] + B), hq * d, dtype)
                      for b in range(batch)]).reshape(batch, B, hq, d)
        kf = np.stack([seq_rows(seed, synth.KIND_KFRESH, b, step[b], range(starts[b], starts[b] + B), hkv * d,
                                dtype) for b in range(batch)]).reshape(batch, B, hkv, d)
        vf = np.stack([seq_rows(seed, synth.KIND_VFRESH, b, step[b], range(starts[b], starts[b] + B), hkv * d,
                                dtype) for b in range(batch)]).reshape(batch, B, hkv, d)
        hid = np.stack([seq_hidden(seed, b, step[b], range(starts[b], starts[b] + B), H, V, sigma, dtype, p_plant)
                        for b in range(batch)])
        kf_dev, vf_dev = dev(kf, dtype), dev(vf, dtype)
        F.fdllm_block_attn_ragged(adesc, _ints(blk), dev(q, dtype), kc_dev, vc_dev, kf_dev, vf_dev, out, None, aws,
                                  ws_bytes=wsb)
        t_before = t_dev.cpu().numpy().astype(np.int64)
        F.fdllm_confidence_select_ragged(sdesc, _ints(starts), dev(hid, dtype), w_dev, t_dev, outs.unmasked,
                                         outs.conf, outs.kappa, outs.argmax, outs.n_left, outs.ws)
        # the fused cache update: each sequence's fresh K/V go to its own window
        F.fdllm_kv_splice_ragged(batch, n, hkv, d, _ints(starts), B, F.BF16, kc_dev, vc_dev, kf_dev, vf_dev)
        got = outs.host()
        assert F.fdllm_last_device_error() == (F.OK, 0)
        o_gpu = out.cpu().numpy().astype(np.float64)
        kc_h = kc_dev.view(torch.int16).cpu().numpy().view(np.uint16)
        for b in range(batch):
            if done[b]:
                continue
            s = starts[b]
            o_ref, _ = O.block_attention(f64(q[b:b + 1], dtype), f64(kc[b:b + 1], dtype), f64(vc[b:b + 1], dtype),
                                         f64(kf[b:b + 1], dtype), f64(vf[b:b + 1], dtype), mode="dual", s=s,
                                         e=s + B, n_q_heads=hq, n_kv_heads=hkv)
            assert_attention_close(o_gpu[b:b + 1], o_ref)
            _, info = O.decode_step(t_before[b:b + 1], f64(hid[b:b + 1], dtype), w64, s=s, block_size=B,
                                    mask_id=V, tau=tau)
            exempt += compare_select(info, {k: v[b:b + 1] for k, v in got.items()}, tau)
            assert np.array_equal(kc_h[b], O.kv_splice(kc[b:b + 1], kf[b:b + 1], s)[0])
        for b in range(batch):                                   # host mirror of the splice
            kc[b] = O.kv_splice(kc[b:b + 1], kf[b:b + 1], starts[b])[0]
            vc[b] = O.kv_splice(vc[b:b + 1], vf[b:b + 1], starts[b])[0]
        # advance: a sequence whose block is decoded moves on and has its cache refreshed
        for b in range(batch):
            if done[b]:
                continue
            step[b] += 1
            steps_in_block[b] += 1
            assert steps_in_block[b] <= B
            if got["n_left"][b] == 0:
                steps_in_block[b] = 0
                if blk[b] + 1 == nblk:
                    done[b] = True
                else:
                    blk[b] += 1
                    advanced += 1
                    kc[b] = seq_cache(seed, synth.KIND_KCACHE, b, n, hkv, d, blk[b], dtype)
                    vc[b] = seq_cache(seed, synth.KIND_VCACHE, b, n, hkv, d, blk[b], dtype)
        kc_dev.copy_(dev(kc, dtype))
        vc_dev.copy_(dev(vc, dtype))
    assert all(done)
    t = t_dev.cpu().numpy()
    assert not (t == V).any() and t.max() < V
    assert np.array_equal(t[:, :prompt_len], tokens0[:, :prompt_len])
    assert advanced == batch * (nblk - 1)
    assert exempt <= 6
    assert apart >= 5          # the oracle alone: 11 of 30 steps


@pytest.mark.parametrize("fp8kv", [False, True])
def test_attention_llada_batch16_full_size_sampled(fp8kv):
    """The DualCache batch-16 LLaDA shape (N = 1024, 32 heads x 128, block 32), sequence b at block b mod 8,
    inputs drawn on the device; three sequences' outputs checked row by row against the oracle (with the
    FP8 cache: over the oracle's dequantisation of the same cache)."""
    b, P, L, B, h, d, seed = 16, 768, 256, 32, 32, 128, 41
    n = P + L
    blocks = [i % (L // B) for i in range(b)]
    kc = torch.empty(b, n, h, d, dtype=torch.bfloat16, device="cuda")
    vc = torch.empty_like(kc)
    F.fdllm_synth_kv_cache(seed, F.SYNTH_KCACHE, b, n, h, d, 0, 1.0, F.BF16, kc)
    F.fdllm_synth_kv_cache(seed, F.SYNTH_VCACHE, b, n, h, d, 0, 1.0, F.BF16, vc)
    # fresh rows: each sequence's own block positions (drawn one sequence at a time on the device)
    q = torch.empty(b, B, h, d, dtype=torch.bfloat16, device="cuda")
    kf, vf = torch.empty(b, B, h, d, dtype=torch.bfloat16, device="cuda"), torch.empty(b, B, h, d, dtype=torch.bfloat16, device="cuda")
    for i, k in enumerate(blocks):
        s = P + k * B
        tmp = torch.empty(i + 1, B, h * d, dtype=torch.bfloat16, device="cuda")
        for kind, dst in ((F.SYNTH_Q, q), (F.SYNTH_KFRESH, kf), (F.SYNTH_VFRESH, vf)):
            F.fdllm_synth_rows(seed, kind, i + 1, 0, s, B, h * d, 1.0, F.BF16, tmp)
            dst[i] = tmp[i].view(B, h, d)
    desc = F.attn_desc(batch=b, prompt_len=P, gen_length=L, block_size=B, block_idx=0, n_q_heads=h, n_kv_heads=h,
                       head_dim=d, use_cache=1, dual_cache=1, dtype=F.BF16, out_f32=1)
    out = torch.empty(b, B, h, d, dtype=torch.float32, device="cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    bidx = _ints(blocks)
    if fp8kv:
        kq = torch.empty(b, n, h, d, dtype=torch.uint8, device="cuda")
        vq = torch.empty_like(kq)
        ks = torch.empty(b, n, h, dtype=torch.float32, device="cuda")
        vs = torch.empty_like(ks)
        F.fdllm_kv_splice_fp8(F.SPLICE_REFRESH, b, n, h, d, 0, n, F.BF16, kq, ks, vq, vs, kc, vc)
        F.fdllm_block_attn_fp8kv(desc, bidx, q, kq, ks, vq, vs, kf, vf, out, None, ws, ws_bytes=0)
    else:
        F.fdllm_block_attn_ragged(desc, bidx, q, kc, vc, kf, vf, out, None, ws, ws_bytes=0)
    torch.cuda.synchronize()
    assert F.fdllm_last_device_error() == (F.OK, 0)
    got = out.cpu().numpy().astype(np.float64)
    per = n * h * d
    for i in (0, 7, 13):
        s = P + blocks[i] * B
        kci = synth.scaled_normals(synth.stream_key(seed, synth.KIND_KCACHE, i, 0), per, 1.0, "bf16")
        vci = synth.scaled_normals(synth.stream_key(seed, synth.KIND_VCACHE, i, 0), per, 1.0, "bf16")
        k64 = f64(kci, "bf16").reshape(1, n, h, d)
        v64 = f64(vci, "bf16").reshape(1, n, h, d)
        if fp8kv:
            k64 = O.dequantize_kv_rows(*O.quantize_kv_rows(k64))
            v64 = O.dequantize_kv_rows(*O.quantize_kv_rows(v64))
        rows = lambda kind, w: np.stack([synth.scaled_normals(synth.stream_key(seed, kind, i, 0, p), w, 1.0, "bf16")
                                         for p in range(s, s + B)])
        qi = f64(rows(synth.KIND_Q, h * d), "bf16").reshape(1, B, h, d)
        kfi = f64(rows(synth.KIND_KFRESH, h * d), "bf16").reshape(1, B, h, d)
        vfi = f64(rows(synth.KIND_VFRESH, h * d), "bf16").reshape(1, B, h, d)
        o_ref, _ = O.block_attention(qi, k64, v64, kfi, vfi, mode="dual", s=s, e=s + B, n_q_heads=h, n_kv_heads=h)
        assert_attention_close(got[i:i + 1], o_ref)
