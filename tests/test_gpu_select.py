"""fdllm_confidence_select against the oracle's decode step."""
import numpy as np
import pytest
import torch

from block_cached_decoding_gb300 import configs
from block_cached_decoding_gb300 import fdllm as F
from block_cached_decoding_gb300 import synth
from gpu_helpers import SelectOutputs, code, compare_select, dev, ensure_built, f64
from oracle import fdllm_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


_W = {}


def weight(seed, V, H, sigma, dtype):
    key = (seed, V, H, sigma, dtype)
    if key not in _W:
        w = synth.lm_head_weight(seed, V, H, sigma, dtype)
        _W[key] = (w, dev(w, dtype), f64(w, dtype))
    return _W[key]


def one_step(*, batch, prompt_len, gen_length, block_size, block_idx, H, V, dtype, tau=0.9, p_plant=0.4,
             sigma=None, seed=0, step=0, premask=None, strategy="threshold", factor=1.0, topk=1):
    sigma = sigma if sigma is not None else float(np.sqrt(0.02))
    n = prompt_len + gen_length
    s, e = O.block_window(prompt_len, block_size, block_idx)
    w, w_dev, w64 = weight(seed, V, H, sigma, dtype)
    hid, _, _ = synth.hidden_states(seed, batch, step, range(s, e), H, V, sigma, dtype, p_plant)
    tokens = np.full((batch, n), V, dtype=np.int64)
    tokens[:, :prompt_len] = synth.prompt_tokens(seed, batch, prompt_len, V)
    tokens[:, :s] = np.where(tokens[:, :s] == V, 7, tokens[:, :s])
    if premask is not None:                        # some block positions already decoded
        tokens[:, s:e] = np.where(premask, V, 5)
    ref_tokens, info = O.decode_step(tokens, f64(hid, dtype), w64, s=s, block_size=block_size, mask_id=V, tau=tau,
                                     strategy=strategy, factor=factor, topk=topk)
    strat = {"threshold": F.SELECT_THRESHOLD, "factor": F.SELECT_FACTOR, "topk": F.SELECT_TOPK}[strategy]
    desc = F.select_desc(batch=batch, seq_len=n, block_start=s, block_size=block_size, hidden=H, vocab=V, mask_id=V,
                         threshold=tau, strategy=strat, factor=factor, topk=topk, dtype=code(dtype))
    t_dev = torch.from_numpy(tokens.astype(np.int32)).cuda()
    outs = SelectOutputs(desc, batch, block_size)
    outs.run(desc, dev(hid, dtype), w_dev, t_dev)
    got = outs.host()
    compare_select(info, got, tau, strategy, factor)
    t_got = t_dev.cpu().numpy()
    # tokens: only this step's unmasked positions changed, to the GPU's argmax
    changed = t_got != tokens
    assert not changed[:, :s].any() and not changed[:, e:].any()
    for b in range(batch):
        for i in np.nonzero(got["unmask"][b])[0]:
            assert t_got[b, s + i] == got["token"][b, i]
    assert np.array_equal(got["n_left"], (t_got[:, s:e] == V).sum(axis=1))
    return info, got


def test_tiny_fp32_first_step():
    wl = configs.TINY
    info, got = one_step(batch=1, prompt_len=64, gen_length=64, block_size=16, block_idx=0, H=wl.hidden,
                         V=wl.vocab, dtype="f32", p_plant=wl.p_plant, sigma=wl.sigma_w, seed=wl.seed)
    assert got["unmask"].sum() >= 1


@pytest.mark.parametrize("tau", [0.5, 0.9, 1.0, 0.0])
def test_bf16_thresholds(tau):
    one_step(batch=2, prompt_len=64, gen_length=64, block_size=32, block_idx=1, H=512, V=5000, dtype="bf16", tau=tau,
             seed=1)


def test_bf16_std_reading_all_fallback():
    info, got = one_step(batch=3, prompt_len=16, gen_length=32, block_size=32, block_idx=0, H=256, V=3001,
                         dtype="bf16", sigma=0.02, seed=2)
    assert np.all(got["unmask"].sum(axis=1) == 1)


def test_partially_decoded_block_and_empty_sequence():
    rng = np.random.default_rng(0)
    pm = rng.random((3, 24)) < 0.4
    pm[1] = False                                  # sequence 1 has nothing left to unmask
    info, got = one_step(batch=3, prompt_len=10, gen_length=48, block_size=24, block_idx=1, H=256, V=2048,
                         dtype="bf16", seed=3, premask=pm)
    assert got["unmask"][1].sum() == 0 and got["n_left"][1] == 0


@pytest.mark.parametrize("strategy,kw", [("factor", dict(factor=1.0)), ("factor", dict(factor=0.3)),
                                         ("topk", dict(topk=2)), ("topk", dict(topk=40))])
def test_strategies(strategy, kw):
    one_step(batch=2, prompt_len=32, gen_length=64, block_size=32, block_idx=0, H=256, V=4096, dtype="bf16", seed=4,
             strategy=strategy, **kw)


@pytest.mark.parametrize("H,V,B", [(64, 2, 1), (192, 1000, 7), (1024, 33333, 48), (256, 70000, 256)])
def test_ragged_shapes(H, V, B):
    one_step(batch=1, prompt_len=3, gen_length=B, block_size=B, block_idx=0, H=H, V=V, dtype="bf16", seed=5)


@pytest.mark.parametrize("batch,B,H,V", [(4, 32, 256, 5000),     # 128 block rows: one row tile
                                         (6, 32, 320, 9001),     # 192 rows: two row tiles
                                         (16, 32, 256, 4097),    # 512 rows: four row tiles
                                         (20, 32, 128, 3000)])   # 640 rows: CUDA-core path
def test_batched_row_tiles(batch, B, H, V):
    rng = np.random.default_rng(batch)
    pm = rng.random((batch, B)) < 0.5
    if batch >= 16:
        pm[4:8] = False          # rows 128..255: a row tile with nothing masked is skipped
    one_step(batch=batch, prompt_len=8, gen_length=B, block_size=B, block_idx=0, H=H, V=V, dtype="bf16",
             seed=6, premask=pm)


@pytest.mark.parametrize("batch,B,H,V", [(32, 4, 128, 200),     # 4 vocabulary splits: 4 selectors, 8 sequences each
                                         (100, 1, 192, 5000),    # 8 selectors, 12-13 sequences each
                                         (160, 2, 128, 3000)])   # 320 rows (clusters of 4), 20 sequences each
def test_many_sequences_per_selector(batch, B, H, V):
    """The last CTAs to finish select: at most 8 of them, and never more than there are CTAs, so
    each may take many sequences."""
    rng = np.random.default_rng(batch + B)
    pm = rng.random((batch, B)) < 0.7
    one_step(batch=batch, prompt_len=5, gen_length=B, block_size=B, block_idx=0, H=H, V=V, dtype="bf16",
             seed=8, premask=pm)


@pytest.mark.parametrize("n_masked,strategy,kw", [(0, "threshold", {}), (1, "threshold", {}), (3, "threshold", {}),
                                                  (9, "factor", dict(factor=0.5)), (32, "topk", dict(topk=5)),
                                                  (32, "threshold", {})])
def test_one_sequence_partly_decoded_blocks(n_masked, strategy, kw):
    """One sequence at every stage of a block (one to 32 masked rows, or none) under each rule: the
    selector takes the masked positions from the flags the LM-head CTA computed at its start."""
    rng = np.random.default_rng(40 + n_masked)
    pm = np.zeros((1, 32), bool)
    pm[0, rng.choice(32, n_masked, replace=False)] = True
    info, got = one_step(batch=1, prompt_len=40, gen_length=64, block_size=32, block_idx=1, H=512, V=20000,
                         dtype="bf16", seed=13, premask=pm, strategy=strategy, **kw)
    assert got["n_left"][0] == n_masked - got["unmask"][0].sum()
    assert (got["token"][0] >= 0).sum() == n_masked


def test_nothing_masked_anywhere():
    info, got = one_step(batch=2, prompt_len=8, gen_length=32, block_size=32, block_idx=0, H=256, V=1000,
                         dtype="bf16", seed=7, premask=np.zeros((2, 32), bool))
    assert got["unmask"].sum() == 0 and np.all(got["n_left"] == 0)


def _select_outputs(desc, hid, w, tokens0, ws):
    out = SelectOutputs(desc, desc.batch, desc.block_size)
    out.ws = ws
    t = tokens0.clone()
    out.run(desc, hid, w, t)
    h = out.host()
    h["tokens"] = t.cpu().numpy()
    return h


def test_workspace_needs_no_initialisation_and_can_be_shared():
    """The workspace holds the ticket words and the softmax partials; whatever it contains on
    entry (all ones, random bytes, another shape's leftovers), the results are the
    same as with a fresh workspace."""
    rng = np.random.default_rng(11)
    shapes = [(2, 32, 512, 5003), (1, 16, 256, 20000), (3, 32, 256, 4096)]
    ws = torch.empty(max(F.fdllm_select_workspace_size(
        F.select_desc(batch=b, seq_len=40 + B, block_start=40, block_size=B, hidden=H, vocab=V, mask_id=V))
        for b, B, H, V in shapes), dtype=torch.uint8, device="cuda")
    for rep in range(2):
        for b, B, H, V in shapes:
            n = 40 + B
            desc = F.select_desc(batch=b, seq_len=n, block_start=40, block_size=B, hidden=H, vocab=V, mask_id=V)
            w_host = synth.lm_head_weight(12, V, H, float(np.sqrt(0.02)), "bf16")
            hid_host, _, _ = synth.hidden_states(12, b, rep, range(40, 40 + B), H, V, float(np.sqrt(0.02)), "bf16", 0.4)
            w, hid = dev(w_host, "bf16"), dev(hid_host, "bf16")
            tokens0 = torch.full((b, n), V, dtype=torch.int32, device="cuda")
            fresh = _select_outputs(desc, hid, w, tokens0, torch.zeros(F.fdllm_select_workspace_size(desc),
                                                                      dtype=torch.uint8, device="cuda"))
            for fill in ("ones", "random", "shared"):
                if fill == "ones":
                    ws.fill_(255)
                elif fill == "random":
                    ws.copy_(torch.from_numpy(rng.integers(0, 256, ws.numel(), dtype=np.uint8)).cuda())
                got = _select_outputs(desc, hid, w, tokens0, ws)
                for key in ("unmask", "token", "n_left", "tokens"):
                    assert np.array_equal(got[key], fresh[key]), (fill, key, b, B, H, V)
                assert np.allclose(got["conf"], fresh["conf"], equal_nan=True, rtol=0, atol=0)


@pytest.mark.parametrize("path", ["bf16", "f32", "fp8"])
def test_exact_ties_take_the_lowest_id(path):
    """Copies of the winning W row at other ids (same 32-column chunk, the next chunk, another
    CTA's vocabulary range, and a lower id for half the rows) give bitwise-equal logits: the token
    must be the lowest id among them (reading R3) on every path, and the confidence counts every
    copy."""
    dtype = "f32" if path == "f32" else "bf16"
    V, H, B = 6000, 256, 8
    sigma = float(np.sqrt(0.02))
    rng = np.random.default_rng(17)
    w = synth.lm_head_weight(21, V, H, sigma, dtype).copy()
    targets = [100 + 650 * i for i in range(B)]            # far apart: the copies never overlap
    lowest = []
    for i, t in enumerate(targets):
        ids = [t + 1, t + 37, t + 420]
        if i % 2:
            ids.append(t - 61)
        for c in ids:
            w[c] = w[t]
        lowest.append(min([t] + ids))
    wf = synth.as_f32(w, dtype)
    z = rng.standard_normal((1, B, H)).astype(np.float32)
    h = (z + 6.0 * wf[targets][None]).astype(np.float32)
    hid = h if dtype == "f32" else synth.f32_to_bf16_bits(h)
    n, s = 64, 32
    tokens = np.full((1, n), V, dtype=np.int64)
    tokens[:, :s] = 3
    desc = F.select_desc(batch=1, seq_len=n, block_start=s, block_size=B, hidden=H, vocab=V, mask_id=V,
                         threshold=0.9, dtype=code(dtype))
    t_dev = torch.from_numpy(tokens.astype(np.int32)).cuda()
    outs = SelectOutputs(desc, 1, B)
    if path == "fp8":
        q = torch.empty(V, H, dtype=torch.uint8, device="cuda")
        sc = torch.empty(V, dtype=torch.float32, device="cuda")
        F.fdllm_quantize_fp8_rows(V, H, F.BF16, dev(w, dtype), q, sc)
        outs.ws = torch.empty(F.fdllm_select_fp8w_workspace_size(desc), dtype=torch.uint8, device="cuda")
        F.fdllm_confidence_select_fp8w(desc, dev(hid, dtype), q, sc, t_dev, outs.unmasked, outs.conf, outs.kappa,
                                       outs.argmax, outs.n_left, outs.ws)
        wc, ws_ = O.quantize_fp8_rows(f64(w, dtype))
        hq, hs = O.quantize_fp8_rows(f64(hid, dtype)[0])
        h64, w64 = O.dequantize_fp8_rows(hq, hs)[None], O.dequantize_fp8_rows(wc, ws_)
    else:
        outs.run(desc, dev(hid, dtype), dev(w, dtype), t_dev)
        h64, w64 = f64(hid, dtype), f64(w, dtype)
    got = outs.host()
    _, info = O.decode_step(tokens, h64, w64, s=s, block_size=B, mask_id=V, tau=0.9)
    assert list(info["token"][0]) == lowest
    assert list(got["token"][0]) == lowest
    assert np.allclose(got["conf"][0], info["conf"][0], atol=1e-3)
    assert np.all(info["conf"][0] <= 1.0 / 4 + 1e-9)        # at least four equal maxima per row
