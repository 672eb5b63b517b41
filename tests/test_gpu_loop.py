"""The GPU block loop in lock step with the oracle (tiny fp32 setting, and a
small bf16 batch).  At every step the oracle evaluates the GPU's current state
(tokens, caches, step inputs); disagreements inside the tolerance bands are
counted and the run continues with the GPU's decision."""
import numpy as np
import pytest
import torch

from block_cached_decoding_gb300 import configs, synth
from block_cached_decoding_gb300 import fdllm as F
from block_cached_decoding_gb300.loop import BlockDecoder
from gpu_helpers import assert_attention_close, compare_select, ensure_built, f64
from oracle import fdllm_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def lockstep(wl, tau, strategy="threshold", refresh_interval=None, topk=1):
    dec = BlockDecoder(wl, tau=tau, strategy={"threshold": F.SELECT_THRESHOLD, "factor": F.SELECT_FACTOR,
                                              "topk": F.SELECT_TOPK}[strategy],
                       refresh_interval=refresh_interval, topk=topk)
    w64 = f64(synth.lm_head_weight(wl.seed, wl.vocab, wl.hidden, wl.sigma_w, wl.dtype), wl.dtype)
    state = {"exempt": 0, "steps": 0, "unmasked": 0}
    caches = {}

    def hook(d, r):
        g, k, s, ep = r.step, r.block, r.block_start, r.epoch
        if ep not in caches:
            caches.clear()
            caches[ep] = [f64(synth.kv_cache(wl.seed, kind, wl.batch, wl.seq_len, wl.n_kv_heads, wl.head_dim, ep,
                                              wl.dtype), wl.dtype) for kind in (synth.KIND_KCACHE, synth.KIND_VCACHE)]
        kc, vc = caches[ep]
        p0, p1 = d.query_range(k)
        pos = range(p0, p1)
        b = wl.batch
        q = synth.per_position(wl.seed, synth.KIND_Q, b, g, pos, wl.n_q_heads * wl.head_dim, wl.dtype)
        kf = synth.per_position(wl.seed, synth.KIND_KFRESH, b, g, pos, wl.n_kv_heads * wl.head_dim, wl.dtype)
        vf = synth.per_position(wl.seed, synth.KIND_VFRESH, b, g, pos, wl.n_kv_heads * wl.head_dim, wl.dtype)
        shp = (b, len(pos), -1, wl.head_dim)
        o_ref, _ = O.block_attention(f64(q, wl.dtype).reshape(shp), kc, vc, f64(kf, wl.dtype).reshape(shp),
                                     f64(vf, wl.dtype).reshape(shp), mode=wl.mode, s=s, e=s + wl.block_size,
                                     n_q_heads=wl.n_q_heads, n_kv_heads=wl.n_kv_heads)
        assert_attention_close(r.attn_out.cpu().numpy().astype(np.float64), o_ref)
        # select: the oracle evaluates the tokens as they were before this step
        t_after = d.tokens.cpu().numpy().astype(np.int64)
        um = r.unmasked.cpu().numpy().astype(bool)
        t_before = t_after.copy()
        t_before[:, s:s + wl.block_size][um] = wl.mask_id
        hid, _, _ = synth.hidden_states(wl.seed, b, g, range(s, s + wl.block_size), wl.hidden, wl.vocab, wl.sigma_w,
                                        wl.dtype, wl.p_plant)
        _, info = O.decode_step(t_before, f64(hid, wl.dtype), w64, s=s, block_size=wl.block_size, mask_id=wl.mask_id,
                                tau=tau, strategy=strategy, topk=topk)
        got = {"unmask": um, "conf": r.conf.cpu().numpy(), "kappa": r.kappa.cpu().numpy(),
               "token": r.argmax.cpu().numpy()}
        state["exempt"] += compare_select(info, got, tau, strategy)
        state["steps"] += 1
        state["unmasked"] += int(um.sum())
        if tau >= 1.0:
            assert np.all(um.sum(axis=1) == info["masked_before"].any(axis=1))

    tokens, steps = dec.run(hook=hook)
    t = tokens.cpu().numpy()
    assert not (t == wl.mask_id).any() and t.max() < wl.vocab
    assert max(steps) <= wl.block_size
    assert state["unmasked"] == wl.batch * wl.gen_length
    return state, steps


@pytest.mark.parametrize("tau", [0.9, 1.0])
def test_tiny_fp32_loop(tau):
    wl = configs.TINY
    state, steps = lockstep(wl, tau)
    if tau >= 1.0:
        assert steps == [wl.block_size] * (wl.gen_length // wl.block_size)
    assert state["exempt"] <= 2


def test_small_bf16_batched_dual_loop():
    wl = configs.LLADA_BATCH.with_(batch=3, prompt_len=40, gen_length=64, block_size=16, n_q_heads=4,
                                   n_kv_heads=2, head_dim=128, hidden=512, vocab=3000)
    state, _ = lockstep(wl, 0.9)
    assert state["exempt"] <= 3


def test_small_bf16_prefix_loop():
    wl = configs.LLADA_STEP.with_(prompt_len=30, gen_length=64, block_size=32, n_q_heads=4, n_kv_heads=4,
                                  head_dim=64, hidden=256, vocab=2000)
    lockstep(wl, 0.9)


def test_refresh_every_two_steps():
    """Cache refreshed every 2 steps inside a block (the LLaDA-V variant): each step's
    attention must read the caches of its own refresh epoch."""
    wl = configs.LLADA_BATCH.with_(batch=2, prompt_len=24, gen_length=32, block_size=16, n_q_heads=4,
                                   n_kv_heads=4, head_dim=64, hidden=256, vocab=1500)
    state, steps = lockstep(wl, 1.0, refresh_interval=2)           # tau = 1: 16 steps per block, 8 refreshes
    assert steps == [16, 16]


def test_factor_strategy_loop():
    wl = configs.TINY.with_(gen_length=32)
    lockstep(wl, 0.9, strategy="factor")


@pytest.mark.parametrize("steps_per_block", [4, 2])
def test_fixed_count_schedule(steps_per_block):
    """LLaDA's baseline schedule with T < B steps per block: a fixed B / T tokens per step (top-k),
    so every block takes exactly T steps and every step unmasks exactly B / T positions."""
    wl = configs.TINY.with_(gen_length=32)
    k = wl.block_size // steps_per_block
    state, steps = lockstep(wl, 0.9, strategy="topk", topk=k)
    assert steps == [steps_per_block] * (wl.gen_length // wl.block_size)
    assert state["unmasked"] == k * state["steps"]


@pytest.mark.parametrize("name", ["tiny-fp32", "bf16-batch3", "bf16-tau1"])
def test_device_driven_loop_matches_the_host_loop(name):
    """Each block as one CUDA-graph while-loop (fdllm_block_loop) gives the host loop's tokens and step
    counts exactly: the same kernels on the same inputs, with the repetition decided on the device.
    Replaying the captured select also replays its workspace tickets' epoch."""
    wl, tau = {
        "tiny-fp32": (configs.TINY, 0.9),
        "bf16-batch3": (configs.LLADA_BATCH.with_(batch=3, prompt_len=40, gen_length=64, block_size=16,
                                                  n_q_heads=4, n_kv_heads=2, head_dim=128, hidden=512, vocab=3000),
                        0.9),
        "bf16-tau1": (configs.LLADA_STEP.with_(prompt_len=30, gen_length=32, block_size=16, n_q_heads=4,
                                               n_kv_heads=4, head_dim=64, hidden=256, vocab=2000, mode="dual"), 1.0),
    }[name]
    t_host, s_host = BlockDecoder(wl, tau=tau).run()
    t_host = t_host.clone()
    t_dev, s_dev = BlockDecoder(wl, tau=tau).run_graph()
    assert s_dev == s_host
    assert torch.equal(t_dev, t_host)
    if tau >= 1.0:
        assert s_dev == [wl.block_size] * (wl.gen_length // wl.block_size)


def test_device_driven_loop_stops_at_the_step_cap():
    wl = configs.LLADA_STEP.with_(prompt_len=30, gen_length=32, block_size=16, n_q_heads=4, n_kv_heads=4,
                                  head_dim=64, hidden=256, vocab=2000, mode="dual")
    with pytest.raises(RuntimeError, match="did not finish within 15 steps"):
        BlockDecoder(wl, tau=1.0).run_graph(max_steps_per_block=15)    # tau = 1: 16 steps per block


@pytest.mark.parametrize("r", [1, 2, 4])
def test_device_loop_refresh_every_r_steps(r):
    """The refresh-every-r-steps cache inside the device-driven loop (a conditional graph node before step
    c of a block whenever r divides c > 0, keyed by the loop's device step counter) gives the host loop's
    tokens and step counts exactly; the host loop is itself checked against the oracle in lock step
    (test_refresh_every_two_steps)."""
    wl = configs.LLADA_BATCH.with_(batch=2, prompt_len=24, gen_length=32, block_size=16, n_q_heads=4, n_kv_heads=4,
                                   head_dim=64, hidden=256, vocab=1500)
    t_host, s_host = BlockDecoder(wl, tau=1.0, refresh_interval=r).run()
    t_host = t_host.clone()
    t_dev, s_dev = BlockDecoder(wl, tau=1.0, refresh_interval=r).run_graph()
    assert s_dev == s_host == [16, 16]
    assert torch.equal(t_dev, t_host)


def test_refresh_every_step_equals_full_attention_on_the_gpu():
    """With the cache refreshed from this step's keys and values at every position (refresh every step,
    r = 1), the DualCache attention of the block equals the no-cache attention over the whole sequence
    at the block's rows (the pages' exactness claim for a fresh cache), up to bf16 rounding of the
    outputs, and both equal the oracle's full attention."""
    b, P, G, B, k, h, d = 2, 40, 64, 16, 2, 4, 128
    n = P + G
    s = P + k * B
    seed, step = 5, 3
    full_k = synth.per_position(seed, synth.KIND_KFRESH, b, step, range(n), h * d, "bf16").reshape(b, n, h, d)
    full_v = synth.per_position(seed, synth.KIND_VFRESH, b, step, range(n), h * d, "bf16").reshape(b, n, h, d)
    q_all = synth.per_position(seed, synth.KIND_Q, b, step, range(n), h * d, "bf16").reshape(b, n, h, d)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    kc, vc = dev(full_k), dev(full_v)                      # the refreshed cache: this step's K/V everywhere
    common = dict(batch=b, prompt_len=P, gen_length=G, block_size=B, block_idx=k, n_q_heads=h, n_kv_heads=h,
                  head_dim=d, dtype=F.BF16, out_f32=1)
    dual = F.attn_desc(use_cache=1, dual_cache=1, **common)
    none = F.attn_desc(use_cache=0, dual_cache=0, **common)
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    o_dual = torch.empty(b, B, h, d, dtype=torch.float32, device="cuda")
    o_full = torch.empty(b, n, h, d, dtype=torch.float32, device="cuda")
    F.fdllm_block_attn(dual, dev(q_all[:, s:s + B]), kc, vc, dev(full_k[:, s:s + B]), dev(full_v[:, s:s + B]), o_dual,
                       None, ws, ws_bytes=0)
    F.fdllm_block_attn(none, dev(q_all), kc, vc, kc, vc, o_full, None, ws, ws_bytes=0)
    torch.cuda.synchronize()
    a, c = o_dual.cpu().numpy().astype(np.float64), o_full.cpu().numpy().astype(np.float64)[:, s:s + B]
    assert_attention_close(a, c)                          # the same keys: equal up to bf16 rounding of P
    f = lambda x: synth.as_f32(x, "bf16").astype(np.float64)
    ref, _ = O.attention_full(f(q_all[:, s:s + B]), f(full_k), f(full_v), h, h)
    assert_attention_close(a, ref)


# ---------------------------------------------------------------------------
# per-sequence blocks: each sequence moves to its next block on its own
# ---------------------------------------------------------------------------

def _ragged_wl():
    return configs.LLADA_BATCH.with_(batch=4, prompt_len=40, gen_length=64, block_size=16, n_q_heads=4,
                                     n_kv_heads=2, head_dim=128, hidden=256, vocab=1500, p_plant=0.3, seed=9)


def test_per_sequence_blocks_host_loop_against_the_oracle():
    """Each sequence moves to its next block as soon as its own block is decoded, its caches then
    recomputed for that block (the per-sequence reading of the batched loop).  At every step the oracle
    evaluates each unfinished sequence at its own block, step and cache epoch: the attention of every
    query row and the select of every masked row."""
    wl, tau = _ragged_wl(), 0.9
    b, B, hq, hkv, d = wl.batch, wl.block_size, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    w64 = f64(synth.lm_head_weight(wl.seed, wl.vocab, wl.hidden, wl.sigma_w, wl.dtype), wl.dtype)
    dec = BlockDecoder(wl, tau=tau, fused_update=True)
    state = {"exempt": 0, "apart": 0, "checked": 0}

    def hook(dd, out, blocks, starts, steps, done):
        state["apart"] += len({blocks[i] for i in range(b) if not done[i]}) > 1
        t_after = dd.tokens.cpu().numpy().astype(np.int64)
        um = dd.unmasked.cpu().numpy().astype(bool)
        got = {"unmask": um, "conf": dd.conf.cpu().numpy(), "kappa": dd.kappa.cpu().numpy(),
               "token": dd.argmax.cpu().numpy()}
        o_gpu = out.cpu().numpy().astype(np.float64)
        for i in range(b):
            if done[i]:
                continue
            s, g, ep = starts[i], steps[i], blocks[i]
            pos = range(s, s + B)
            kc = f64(synth.kv_cache(wl.seed, synth.KIND_KCACHE, b, wl.seq_len, hkv, d, ep, wl.dtype), wl.dtype)[i:i + 1]
            vc = f64(synth.kv_cache(wl.seed, synth.KIND_VCACHE, b, wl.seq_len, hkv, d, ep, wl.dtype), wl.dtype)[i:i + 1]
            q = f64(synth.per_position(wl.seed, synth.KIND_Q, b, g, pos, hq * d, wl.dtype), wl.dtype)[i:i + 1]
            kf = f64(synth.per_position(wl.seed, synth.KIND_KFRESH, b, g, pos, hkv * d, wl.dtype), wl.dtype)[i:i + 1]
            vf = f64(synth.per_position(wl.seed, synth.KIND_VFRESH, b, g, pos, hkv * d, wl.dtype), wl.dtype)[i:i + 1]
            o_ref, _ = O.block_attention(q.reshape(1, B, hq, d), kc, vc, kf.reshape(1, B, hkv, d),
                                         vf.reshape(1, B, hkv, d), mode="dual", s=s, e=s + B, n_q_heads=hq,
                                         n_kv_heads=hkv)
            assert_attention_close(o_gpu[i:i + 1], o_ref)
            t_before = t_after[i:i + 1].copy()
            t_before[:, s:s + B][um[i:i + 1]] = wl.mask_id
            hid, _, _ = synth.hidden_states(wl.seed, b, g, pos, wl.hidden, wl.vocab, wl.sigma_w, wl.dtype, wl.p_plant)
            _, info = O.decode_step(t_before, f64(hid, wl.dtype)[i:i + 1], w64, s=s, block_size=B,
                                    mask_id=wl.mask_id, tau=tau)
            state["exempt"] += compare_select(info, {k: v[i:i + 1] for k, v in got.items()}, tau)
            state["checked"] += 1

    tokens, steps = dec.run_ragged(hook=hook)
    t = tokens.cpu().numpy()
    assert not (t == wl.mask_id).any() and t.max() < wl.vocab
    assert all(n <= wl.gen_length for n in steps)
    assert state["apart"] >= 3                     # the sequences were at different blocks at times
    assert state["exempt"] <= 2 + 0.01 * state["checked"] * B


@pytest.mark.parametrize("tau", [0.9, 1.0])
def test_per_sequence_device_loop_matches_the_host_loop(tau):
    """The whole per-sequence generation as one CUDA-graph while-loop (fdllm_block_loop_create_ragged:
    each sequence's block index, window start and step advanced on the device, the moved sequences'
    caches refreshed in a conditional node) gives the host loop's tokens and per-sequence step counts
    exactly."""
    wl = _ragged_wl()
    t_host, s_host = BlockDecoder(wl, tau=tau, fused_update=True).run_ragged()
    t_host = t_host.clone()
    dec = BlockDecoder(wl, tau=tau, fused_update=True)
    t_dev, s_dev = dec.run_ragged_graph()
    assert s_dev == s_host
    assert torch.equal(t_dev, t_host)
    assert dec.rg["block_idx"].tolist() == [wl.gen_length // wl.block_size - 1] * wl.batch
    if tau >= 1.0:
        assert s_dev == [wl.gen_length] * wl.batch    # one position per step, every sequence
    t_again, s_again = dec.run_ragged_graph()          # a second launch of a fresh loop starts over
    assert s_again == s_host and torch.equal(t_again, t_host)
