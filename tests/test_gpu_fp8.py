"""FP8 weight cache on the GPU: the per-row E4M3 quantiser is bit-exact against the
oracle's (codes and scales), and fdllm_confidence_select_fp8w matches the oracle's
decode step on the same quantised operands (the tolerance rules of the bf16 path)."""
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


def gpu_quantize(x_dev, dtype):
    rows, cols = x_dev.shape
    q = torch.empty(rows, cols, dtype=torch.uint8, device="cuda")
    s = torch.empty(rows, dtype=torch.float32, device="cuda")
    F.fdllm_quantize_fp8_rows(rows, cols, code(dtype), x_dev, q, s)
    torch.cuda.synchronize()
    return q, s


def special_rows(cols, rng):
    """Rows that probe the rounding and the scale rule: an all-zero row, exact E4M3 midpoints after
    scaling (ties to even), a row whose maximum is exactly 448 * 2^k, values far below the
    smallest subnormal, negative zeros, and large and small magnitudes."""
    grid = O.e4m3_decode(np.array([c for c in range(128) if c != 0x7F], dtype=np.uint8))
    mids = (grid[:-1] + grid[1:]) / 2
    rows = [np.zeros(cols)]
    r = rng.choice(mids, cols) * rng.choice([-1.0, 1.0], cols)
    r[0] = 448.0                                      # scale 1: the midpoints stay midpoints
    rows.append(r)
    r = rng.choice(mids, cols) * 2.0 ** -5
    r[1] = 448.0 * 2.0 ** -5                          # scale 2^-5, still exact
    rows.append(r)
    r = rng.standard_normal(cols) * 1e-6
    r[2] = 1.0                                        # most values round to (signed) zero
    rows.append(r)
    r = -np.abs(rng.standard_normal(cols)) * 0.0
    r[3] = -3.0
    rows.append(r)
    rows.append(rng.standard_normal(cols) * 3e4)
    rows.append(rng.standard_normal(cols) * 3e-3)
    return np.stack(rows)


@pytest.mark.parametrize("dtype,rows,cols", [("f32", 37, 100), ("bf16", 300, 256), ("f32", 2000, 64),
                                             ("bf16", 5, 4096)])
def test_quantize_rows_bit_exact(dtype, rows, cols):
    rng = np.random.default_rng(rows + cols)
    x = rng.standard_normal((rows, cols)) * np.exp2(rng.integers(-20, 20, (rows, 1)))
    x = np.concatenate([special_rows(cols, rng), x])
    stored = x.astype(np.float32) if dtype == "f32" else synth.f32_to_bf16_bits(x.astype(np.float32))
    q, s = gpu_quantize(dev(stored, dtype), dtype)
    want_q, want_s = O.quantize_fp8_rows(f64(stored, dtype))
    got_q = q.cpu().numpy()
    assert np.array_equal(s.cpu().numpy().astype(np.float64), want_s)
    bad = np.argwhere(got_q != want_q)
    assert len(bad) == 0, (bad[:5], got_q[tuple(bad[0])], want_q[tuple(bad[0])])


def test_quantize_nothing_to_do():
    F.fdllm_quantize_fp8_rows(0, 64, F.BF16, None, None, None)
    F.fdllm_quantize_fp8_rows(4, 0, F.BF16, None, None, None)


_W = {}


def fp8_weight(seed, V, H, sigma):
    """bf16 W drawn by the generator, its FP8 cache made on the GPU and checked against the
    oracle's codes, and the oracle's dequantised float64 W."""
    key = (seed, V, H, sigma)
    if key not in _W:
        _W.clear()
        w = synth.lm_head_weight(seed, V, H, sigma, "bf16")
        q, s = gpu_quantize(dev(w, "bf16"), "bf16")
        want_q, want_s = O.quantize_fp8_rows(f64(w, "bf16"))
        assert np.array_equal(q.cpu().numpy(), want_q) and np.array_equal(s.cpu().numpy(), want_s)
        _W[key] = (q, s, O.dequantize_fp8_rows(want_q, want_s))
    return _W[key]


def fp8_step(*, batch, prompt_len, gen_length, block_size, block_idx, H, V, tau=0.9, p_plant=0.4, seed=0, step=0,
             premask=None, strategy="threshold", factor=1.0, topk=1):
    sigma = float(np.sqrt(0.02))
    n = prompt_len + gen_length
    s, e = O.block_window(prompt_len, block_size, block_idx)
    wq, ws, w64 = fp8_weight(seed, V, H, sigma)
    hid, _, _ = synth.hidden_states(seed, batch, step, range(s, e), H, V, sigma, "bf16", p_plant)
    tokens = np.full((batch, n), V, dtype=np.int64)
    tokens[:, :prompt_len] = synth.prompt_tokens(seed, batch, prompt_len, V)
    tokens[:, :s] = np.where(tokens[:, :s] == V, 7, tokens[:, :s])
    if premask is not None:
        tokens[:, s:e] = np.where(premask, V, 5)
    # the oracle: hidden rows quantised per row, both operands at their exact FP8 values
    hq, hs = O.quantize_fp8_rows(f64(hid, "bf16").reshape(batch * block_size, H))
    h64 = O.dequantize_fp8_rows(hq, hs).reshape(batch, block_size, H)
    _, info = O.decode_step(tokens, h64, w64, s=s, block_size=block_size, mask_id=V, tau=tau, strategy=strategy,
                            factor=factor, topk=topk)
    strat = {"threshold": F.SELECT_THRESHOLD, "factor": F.SELECT_FACTOR, "topk": F.SELECT_TOPK}[strategy]
    desc = F.select_desc(batch=batch, seq_len=n, block_start=s, block_size=block_size, hidden=H, vocab=V, mask_id=V,
                         threshold=tau, strategy=strat, factor=factor, topk=topk, dtype=F.BF16)
    t_dev = torch.from_numpy(tokens.astype(np.int32)).cuda()
    outs = SelectOutputs(desc, batch, block_size)
    outs.ws = torch.empty(F.fdllm_select_fp8w_workspace_size(desc), dtype=torch.uint8, device="cuda")
    F.fdllm_confidence_select_fp8w(desc, dev(hid, "bf16"), wq, ws, t_dev, outs.unmasked, outs.conf, outs.kappa,
                                   outs.argmax, outs.n_left, outs.ws)
    got = outs.host()
    assert F.fdllm_last_device_error() == (F.OK, 0)
    exempt = compare_select(info, got, tau, strategy, factor)
    t_got = t_dev.cpu().numpy()
    changed = t_got != tokens
    assert not changed[:, :s].any() and not changed[:, e:].any()
    for b in range(batch):
        for i in np.nonzero(got["unmask"][b])[0]:
            assert t_got[b, s + i] == got["token"][b, i]
    assert np.array_equal(got["n_left"], (t_got[:, s:e] == V).sum(axis=1))
    return info, got, exempt


@pytest.mark.parametrize("batch,B,H,V", [
    (1, 32, 256, 5000),      # one 128-row tile, clusters of one
    (1, 7, 128, 3001),       # ragged block, vocabulary not a multiple of the 64-row unit
    (4, 32, 512, 20000),     # 128 block rows, quantised by the LM-head kernel itself (a CTA per row)
    (4, 32, 128, 2000),      # 128 rows but only 32 vocabulary splits: the row quantiser kernel first
    (8, 32, 256, 3000),      # 256 rows: clusters of two sharing each W tile
    (16, 32, 128, 2000),     # 512 rows: clusters of four
])
def test_select_fp8w_matches_oracle(batch, B, H, V):
    fp8_step(batch=batch, prompt_len=40, gen_length=4 * B, block_size=B, block_idx=1, H=H, V=V)


@pytest.mark.parametrize("tau", [0.5, 1.0])
def test_select_fp8w_thresholds(tau):
    _, got, _ = fp8_step(batch=2, prompt_len=30, gen_length=64, block_size=32, block_idx=0, H=256, V=4000, tau=tau)
    if tau >= 1.0:
        assert np.all(got["unmask"].sum(axis=1) == 1)


def test_select_fp8w_partly_decoded_and_topk():
    rng = np.random.default_rng(3)
    premask = rng.random((3, 16)) < 0.5
    premask[2] = False                                # a sequence with nothing left to decode
    fp8_step(batch=3, prompt_len=20, gen_length=32, block_size=16, block_idx=1, H=256, V=2500, premask=premask,
             strategy="topk", topk=3)


def test_select_fp8w_llada_step_full_size():
    """The benchmarked LLaDA-8B step (V = 126464, H = 4096, one block of 32) through the FP8
    cache: every masked row against the oracle."""
    from fullsize_helpers import weight_f64
    wl = configs.LLADA_STEP
    V, H, B = wl.vocab, wl.hidden, wl.block_size
    w = torch.empty(V, H, dtype=torch.bfloat16, device="cuda")
    F.fdllm_synth_normals(wl.seed, F.SYNTH_W, [], V * H, 0, wl.sigma_w, F.BF16, w)
    q, s = gpu_quantize(w, "bf16")
    del w
    w_stored = weight_f64(wl.seed, V, H, wl.sigma_w)
    want_q, want_s = O.quantize_fp8_rows(w_stored)
    assert np.array_equal(s.cpu().numpy(), want_s)
    assert np.array_equal(q.cpu().numpy(), want_q)
    w64 = O.dequantize_fp8_rows(want_q, want_s)
    del want_q
    n = wl.seq_len
    st, e = O.block_window(wl.prompt_len, B, 0)
    hid = torch.empty(1, B, H, dtype=torch.bfloat16, device="cuda")
    wb = torch.empty(V, H, dtype=torch.bfloat16, device="cuda")
    F.fdllm_synth_normals(wl.seed, F.SYNTH_W, [], V * H, 0, wl.sigma_w, F.BF16, wb)
    F.fdllm_synth_hidden(wl.seed, 1, 0, st, B, H, V, wl.p_plant, wb, F.BF16, hid)
    del wb
    tokens = np.full((1, n), wl.mask_id, dtype=np.int64)
    tokens[:, :wl.prompt_len] = synth.prompt_tokens(wl.seed, 1, wl.prompt_len, V)
    hid_host = hid.float().cpu().numpy().astype(np.float64).reshape(B, H)
    hq, hs = O.quantize_fp8_rows(hid_host)
    _, info = O.decode_step(tokens, O.dequantize_fp8_rows(hq, hs)[None], w64, s=st, block_size=B,
                            mask_id=wl.mask_id, tau=wl.taus[0])
    desc = F.select_desc(batch=1, seq_len=n, block_start=st, block_size=B, hidden=H, vocab=V, mask_id=wl.mask_id,
                         threshold=wl.taus[0], dtype=F.BF16)
    t_dev = torch.from_numpy(tokens.astype(np.int32)).cuda()
    outs = SelectOutputs(desc, 1, B)
    outs.ws = torch.empty(F.fdllm_select_fp8w_workspace_size(desc), dtype=torch.uint8, device="cuda")
    F.fdllm_confidence_select_fp8w(desc, hid, q, s, t_dev, outs.unmasked, outs.conf, outs.kappa, outs.argmax,
                                   outs.n_left, outs.ws)
    got = outs.host()
    assert F.fdllm_last_device_error() == (F.OK, 0)
    assert compare_select(info, got, wl.taus[0]) <= 2
