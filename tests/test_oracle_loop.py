"""Pins for the oracle's block loop (section 3.4.4, Algorithm 1) on the tiny setting."""
import numpy as np
import pytest

from block_cached_decoding_gb300 import configs, synth
from oracle import fdllm_oracle as O


def _setup(wl, sigma_w=None):
    sw = wl.sigma_w if sigma_w is None else sigma_w
    w = synth.lm_head_weight(wl.seed, wl.vocab, wl.hidden, sw, wl.dtype)
    w64 = synth.as_f32(w, wl.dtype).astype(np.float64)

    def hidden_fn(g, s, tokens):
        rows, _, _ = synth.hidden_states(wl.seed, wl.batch, g, range(s, s + wl.block_size), wl.hidden,
                                         wl.vocab, sw, wl.dtype, wl.p_plant)
        return synth.as_f32(rows, wl.dtype).astype(np.float64)

    prompt = synth.prompt_tokens(wl.seed, wl.batch, wl.prompt_len, wl.vocab)
    return w64, hidden_fn, prompt


@pytest.mark.parametrize("tau", [0.9, 1.0])
def test_tiny_loop_progress_and_step_counts(tau):
    wl = configs.TINY.with_(batch=2)
    w64, hidden_fn, prompt = _setup(wl)
    seen = []

    def hook(g, k, s, tokens, info):
        # every unmasked token is the step's argmax, and at least one unmasks per sequence
        # that still had a masked position
        for b in range(wl.batch):
            assert (info["unmask"][b].sum() >= 1) == bool(info["masked_before"][b].any())
            for i in np.nonzero(info["unmask"][b])[0]:
                assert tokens[b, s + i] == info["token"][b, i]
        if tau >= 1.0:
            assert np.all(info["unmask"].sum(axis=1) == info["masked_before"].any(axis=1))
        seen.append(g)
        return tokens

    tokens, rec = O.generate(prompt, gen_length=wl.gen_length, block_size=wl.block_size, mask_id=wl.mask_id,
                             tau=tau, w=w64, hidden_fn=hidden_fn, step_hook=hook)
    assert not (tokens == wl.mask_id).any()
    assert np.array_equal(tokens[:, :wl.prompt_len], prompt)
    assert tokens.max() < wl.vocab
    blocks = wl.gen_length // wl.block_size
    per_block = np.bincount([r["block"] for r in rec], minlength=blocks)
    assert per_block.max() <= wl.block_size
    if tau >= 1.0:
        assert len(rec) == wl.gen_length and np.all(per_block == wl.block_size)
    else:
        assert len(rec) < wl.gen_length                 # parallel steps happen


def test_planted_rows_predict_their_target():
    wl = configs.TINY
    w64, _, _ = _setup(wl)
    pos = range(64, 80)
    rows, planted, target = synth.hidden_states(wl.seed, 1, 3, pos, wl.hidden, wl.vocab, wl.sigma_w, wl.dtype, wl.p_plant)
    st = O.lm_head_confidence(synth.as_f32(rows[0], wl.dtype).astype(np.float64), w64)
    assert planted.sum() >= 3
    assert np.all(st["token"][planted[0]] == target[0][planted[0]])
    assert np.all(st["conf"][planted[0]] > 0.99)


def test_std_reading_gives_all_fallback_steps():
    """With sigma_W read as a standard deviation, confidences stay low and tau = 0.9 never fires."""
    wl = configs.TINY
    w64, hidden_fn, prompt = _setup(wl, sigma_w=wl.sigma_w_alt)
    tokens, rec = O.generate(prompt, gen_length=32, block_size=wl.block_size, mask_id=wl.mask_id,
                             tau=0.9, w=w64, hidden_fn=hidden_fn)
    assert all(r["n_unmasked"] == 1 for r in rec) and len(rec) == 32


@pytest.mark.parametrize("T", [1, 2, 4, 16])
def test_fixed_count_schedule_takes_T_steps_per_block(T):
    """LLaDA's baseline schedule (fixed B / T tokens per step) as top-k selection: every block ends
    in exactly T steps, each step unmasks B / T positions per sequence, and they are the B / T most
    confident of the masked ones."""
    wl = configs.TINY.with_(batch=2)
    w64, hidden_fn, prompt = _setup(wl)
    k = wl.block_size // T

    def hook(g, blk, s, tokens, info):
        for b in range(wl.batch):
            sel = np.nonzero(info["unmask"][b])[0]
            assert len(sel) == k
            rest = [i for i in np.nonzero(info["masked_before"][b])[0] if i not in sel]
            if rest:                                  # every pick at least as confident as every non-pick
                assert info["conf"][b, sel].min() >= info["conf"][b, rest].max()
        return tokens

    tokens, rec = O.generate(prompt, gen_length=wl.gen_length, block_size=wl.block_size, mask_id=wl.mask_id,
                             tau=0.9, w=w64, hidden_fn=hidden_fn, strategy="topk", topk=k, step_hook=hook)
    per_block = np.bincount([r["block"] for r in rec], minlength=wl.gen_length // wl.block_size)
    assert np.all(per_block == T)
    assert not (tokens == wl.mask_id).any()
