"""Plain float64 CPU oracle for Fast-dLLM block-cached decoding (test infrastructure).

This module is test infrastructure.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import or call it; the product
path (the CUDA library and its binding) never does, and shares no code with it.

Every function states the passage of the Fast-dLLM pages it follows.  Pages:

* "Fast-dLLM ... paper-graph-ui summary": section 3.2 (architecture), 3.4.2
  (approximate KV cache: PrefixCache, DualCache, block-wise scheme, fused
  updates), 3.4.3 (confidence, Theorem 1, threshold and factor strategies, the
  three-line PyTorch idiom), 3.4.4 (the integrated Algorithm 1 loop).
* "NVlabs/Fast-dLLM" README: the knobs gen_length, block_size, use_cache,
  if_cache_position (dual cache), threshold.

Inputs are the exact stored values (bfloat16 or float32) upcast to float64.
Readings where the pages are silent:

* R1 strict ``c > tau`` (the pages write both ">= tau" and "exceeds tau").
* R2 ranking for the fallback uses kappa = log((1 - c) / c), strictly
  decreasing in c, evaluated without cancellation so saturated confidences
  (c == 1.0 in floating point) still order correctly.
* R3 ties: lowest vocabulary id for the argmax; lowest position for the
  fallback pick.
* R4 softmax scale 1/sqrt(head_dim); no causal mask (bidirectional).
* R5 PrefixCache queries are the block *and* the suffix positions [s, N).
* R6 batched decoding runs in lock step over a shared block index; with
  per-sequence blocks each sequence is this oracle run alone at its own window.
* R13 FP8 weight cache: E4M3 codes, one power-of-two scale per row, round to
  nearest even; hidden rows quantised the same way per step.
* R14 FP8 KV cache: cached K and V rows (sequence, position, KV head) stored by
  the R13 rule; attention reads the dequantised cache, fresh K/V unchanged.
"""
from __future__ import annotations

import math

import numpy as np


# ---------------------------------------------------------------------------
# a2: block attention (paper-graph-ui summary, 3.4.2 "PrefixCache", "DualCache";
#     3.4.4 "Per-Block Loop Structure": cached KV outside [s, e), fresh inside)
# ---------------------------------------------------------------------------

def query_positions(mode: str, s: int, e: int, seq_len: int) -> range:
    """Positions whose queries are computed in one step.

    DualCache recomputes only the current block [s, e); PrefixCache recomputes the
    block and every suffix position [s, N); no cache recomputes all of [0, N)."""
    if mode == "dual":
        return range(s, e)
    if mode == "prefix":
        return range(s, seq_len)
    if mode == "none":
        return range(0, seq_len)
    raise ValueError(mode)


def assemble_keys(mode, s, e, cache, fresh):
    """The key (or value) set a step attends to, as one [b, N, Hkv, d] array.

    Positions with fresh projections this step take them from `fresh` (which is
    indexed like the query positions); every other position is read from the
    cache: prefix [0, s) and, for DualCache, suffix [e, N)."""
    b, n = cache.shape[:2]
    out = cache.copy()
    pos = query_positions(mode, s, e, n)
    out[:, pos.start:pos.stop] = fresh
    return out


def attention_full(q, k, v, n_q_heads, n_kv_heads, sm_scale=None):
    """softmax(q k^T * scale) v per (batch, query head); bidirectional, no mask.

    q [b, nq, Hq, d], k/v [b, N, Hkv, d] -> (O [b, nq, Hq, d], lse [b, nq, Hq]).
    Query head h reads key/value head h // (Hq / Hkv) (grouped-query sharing)."""
    b, nq, hq, d = q.shape
    assert hq == n_q_heads and k.shape[2] == n_kv_heads
    group = n_q_heads // n_kv_heads
    scale = 1.0 / math.sqrt(d) if sm_scale is None else sm_scale
    o = np.zeros((b, nq, hq, d))
    lse = np.zeros((b, nq, hq))
    for bi in range(b):
        for h in range(hq):
            kh = k[bi, :, h // group, :]
            vh = v[bi, :, h // group, :]
            scores = (q[bi, :, h, :] @ kh.T) * scale          # [nq, N]
            m = scores.max(axis=1, keepdims=True)
            p = np.exp(scores - m)
            denom = p.sum(axis=1, keepdims=True)
            o[bi, :, h, :] = (p @ vh) / denom
            lse[bi, :, h] = m[:, 0] + np.log(denom[:, 0])
    return o, lse


def block_attention(q, k_cache, v_cache, k_fresh, v_fresh, *, mode, s, e,
                    n_q_heads, n_kv_heads, sm_scale=None):
    """One denoising step's attention for the recomputed queries.

    q [b, nq, Hq, d] and k_fresh / v_fresh [b, nq, Hkv, d] hold the positions
    given by `query_positions(mode, s, e, N)`; caches are [b, N, Hkv, d]."""
    k = assemble_keys(mode, s, e, k_cache, k_fresh)
    v = assemble_keys(mode, s, e, v_cache, v_fresh)
    return attention_full(q, k, v, n_q_heads, n_kv_heads, sm_scale)


# ---------------------------------------------------------------------------
# a8: cache splice / refresh (3.4.2 "Cache Overhead and Fused Updates";
#     3.4.4 step 3 "Cache update")
# ---------------------------------------------------------------------------

def kv_splice(cache, src, start):
    """cache[:, start:start+len] <- src (len = src.shape[1]); returns a new array."""
    out = cache.copy()
    out[:, start:start + src.shape[1]] = src
    return out


# ---------------------------------------------------------------------------
# a3-a5: LM head and confidence (3.4.3 "The Core Idea": c_i = max_v p(x_i = v);
#        the idiom logits.softmax(-1).max(-1))
# ---------------------------------------------------------------------------

def lm_head_confidence(h, w):
    """Confidence statistics of each row of h [R, H] against the vocabulary W [V, H].

    logits l = h W^T.  Returns a dict of float64 / int64 arrays over rows:
      token  lowest index v with l_v = max l (reading R3)
      conf   c = max_v softmax(l)_v = 1 / sum_v exp(l_v - max l)
      kappa  log((1 - c) / c) = log sum_{v != token} exp(l_v - max l), evaluated as
             (m2 - m1) + log sum_{v != token} exp(l_v - m2) with m2 the largest
             logit other than the argmax, so it stays finite when c rounds to 1
      gap    m1 - m2, the top-2 logit gap
    """
    logits = h @ w.T
    r, v = logits.shape
    token = np.argmax(logits, axis=1)                     # first index of the max
    m1 = logits[np.arange(r), token]
    conf = 1.0 / np.exp(logits - m1[:, None]).sum(axis=1)
    kappa = np.full(r, -np.inf)
    gap = np.full(r, np.inf)
    if v > 1:
        rest = logits.copy()
        rest[np.arange(r), token] = -np.inf
        m2 = rest.max(axis=1)
        s2 = np.exp(rest - m2[:, None]).sum(axis=1)
        kappa = (m2 - m1) + np.log(s2)
        gap = m1 - m2
    return {"token": token.astype(np.int64), "conf": conf, "kappa": kappa, "gap": gap, "logits": logits}


def threshold_log_odds(tau: float) -> float:
    """kappa threshold equivalent to c > tau: c > tau <=> kappa < log((1 - tau) / tau); none for tau >= 1."""
    if tau >= 1.0:
        return -math.inf
    if tau <= 0.0:
        return math.inf
    return math.log((1.0 - tau) / tau)


# ---------------------------------------------------------------------------
# a6: selection (3.4.3 "From Theorem to Practice: Threshold Strategy" and the
#     progress guarantee; "Factor Strategy"; fixed top-k of the LLaDA baseline
#     from 5 "Baselines")
# ---------------------------------------------------------------------------

def _fallback(kappa, masked):
    """The single masked position of highest confidence (lowest kappa, lowest index on ties)."""
    best = -1
    for i in range(len(masked)):
        if masked[i] and (best < 0 or kappa[i] < kappa[best]):
            best = i
    return best


def threshold_select(conf, kappa, masked, tau):
    """Unmask every masked position with c_i > tau; if none qualifies and some
    position is masked, unmask the single most confident one.  Returns bool [B]."""
    sel = np.array([bool(masked[i]) and conf[i] > tau for i in range(len(masked))])
    if not sel.any() and np.any(masked):
        sel[_fallback(kappa, masked)] = True
    return sel


def factor_select(kappa, masked, factor):
    """Sort masked positions by confidence (descending); unmask the largest n with
    (n + 1) * (1 - c_(n)) < f, at least one.  1 - c = 1 / (1 + exp(-kappa))."""
    idx = [i for i in range(len(masked)) if masked[i]]
    sel = np.zeros(len(masked), dtype=bool)
    if not idx:
        return sel
    order = sorted(idx, key=lambda i: (kappa[i], i))
    n_best = 0
    for n in range(1, len(order) + 1):
        eps = 1.0 / (1.0 + math.exp(-kappa[order[n - 1]])) if kappa[order[n - 1]] > -700 else 0.0
        if (n + 1) * eps < factor:
            n_best = n
    n_best = max(n_best, 1)
    for i in order[:n_best]:
        sel[i] = True
    return sel


def topk_select(kappa, masked, k):
    """Unmask the k most confident masked positions (all of them if fewer remain)."""
    idx = sorted([i for i in range(len(masked)) if masked[i]], key=lambda i: (kappa[i], i))
    sel = np.zeros(len(masked), dtype=bool)
    for i in idx[:k]:
        sel[i] = True
    return sel


# ---------------------------------------------------------------------------
# a1, a5-a7: one step of the block loop and the whole loop (3.2 "Information
# flow"; 3.4.4 "Per-Block Loop Structure"; Algorithm 1)
# ---------------------------------------------------------------------------

def block_window(prompt_len, block_size, k):
    """Block k (0-based) spans [s, e) with s = |p0| + k B, e = s + B."""
    s = prompt_len + k * block_size
    return s, s + block_size


def decode_step(tokens, hidden_rows, w, *, s, block_size, mask_id, tau,
                strategy="threshold", factor=1.0, topk=1):
    """One confidence-aware unmask step over the block [s, s + B) of every sequence.

    tokens int [b, N] (modified copy returned); hidden_rows [b, B, H] float64 for
    all block positions (rows of unmasked positions are ignored).
    Returns (tokens, info) with per-(b, i) conf / kappa / token / gap (NaN where
    not masked), the unmask mask and the count left masked per sequence."""
    tokens = tokens.copy()
    b = tokens.shape[0]
    B = block_size
    info = {k: np.full((b, B), np.nan) for k in ("conf", "kappa", "gap")}
    info["token"] = np.full((b, B), -1, dtype=np.int64)
    info["unmask"] = np.zeros((b, B), dtype=bool)
    info["masked_before"] = tokens[:, s:s + B] == mask_id
    for bi in range(b):
        masked = info["masked_before"][bi]
        rows = np.nonzero(masked)[0]
        if len(rows) == 0:
            continue
        st = lm_head_confidence(hidden_rows[bi, rows], w)
        for key in ("conf", "kappa", "gap"):
            info[key][bi, rows] = st[key]
        info["token"][bi, rows] = st["token"]
        kap = np.where(masked, info["kappa"][bi], np.inf)
        cf = np.where(masked, info["conf"][bi], -np.inf)
        if strategy == "threshold":
            sel = threshold_select(cf, kap, masked, tau)
        elif strategy == "factor":
            sel = factor_select(kap, masked, factor)
        elif strategy == "topk":
            sel = topk_select(kap, masked, topk)
        else:
            raise ValueError(strategy)
        info["unmask"][bi] = sel
        for i in np.nonzero(sel)[0]:
            tokens[bi, s + i] = info["token"][bi, i]
    info["n_masked_left"] = (tokens[:, s:s + B] == mask_id).sum(axis=1)
    return tokens, info


def generate(prompt, *, gen_length, block_size, mask_id, tau, w, hidden_fn,
             strategy="threshold", factor=1.0, topk=1, step_hook=None, max_steps_per_block=None):
    """Block-wise generation (Algorithm 1), lock-step over the batch.

    x = [prompt; MASK x L]; for each block left to right, run unmask steps until
    no position of the block is masked in any sequence.  `hidden_fn(g, s, tokens)`
    returns the float64 hidden rows [b, B, H] of step g (the synthetic stand-in for
    the model forward pass).  `step_hook(g, k, s, tokens, info)` may inspect or
    replace the tokens after each step (returns tokens).
    Returns (tokens, per-step records)."""
    b, p = prompt.shape
    n = p + gen_length
    assert gen_length % block_size == 0
    tokens = np.full((b, n), mask_id, dtype=np.int64)
    tokens[:, :p] = prompt
    records = []
    g = 0
    for k in range(gen_length // block_size):
        s, e = block_window(p, block_size, k)
        steps = 0
        while (tokens[:, s:e] == mask_id).any():
            h = hidden_fn(g, s, tokens)
            tokens, info = decode_step(tokens, h, w, s=s, block_size=block_size, mask_id=mask_id,
                                       tau=tau, strategy=strategy, factor=factor, topk=topk)
            if step_hook is not None:
                tokens = step_hook(g, k, s, tokens, info)
            records.append({"step": g, "block": k, "n_unmasked": int(info["unmask"].sum()),
                            "per_seq": info["unmask"].sum(axis=1)})
            g += 1
            steps += 1
            cap = max_steps_per_block or block_size
            assert steps <= cap, "a block must finish within block_size steps"
    return tokens, records


# ---------------------------------------------------------------------------
# Theorem 1 (3.4.3): product of marginals versus the joint
# ---------------------------------------------------------------------------

def marginals(p_joint):
    """Per-position marginals of a joint table p[x_1, ..., x_n]."""
    n = p_joint.ndim
    return [p_joint.sum(axis=tuple(a for a in range(n) if a != j)) for j in range(n)]


def product_of_marginals(p_joint):
    """q(x) = prod_j p_j(x_j) as a table of the joint's shape."""
    q = np.ones(())
    for m in marginals(p_joint):
        q = np.multiply.outer(q, m)
    return q


def greedy(table):
    """argmax of a table as an index tuple (first in C order on ties)."""
    return tuple(int(i) for i in np.unravel_index(int(np.argmax(table)), table.shape))


def kv_cache_bytes(seq_len, layers, heads, head_dim, bytes_per_elem):
    """Key plus value cache size (section 6, Limitation 6): N x layers x heads x d x 2 (K and V) x bytes."""
    return seq_len * layers * heads * head_dim * 2 * bytes_per_elem


# ---------------------------------------------------------------------------
# f4: FP8 weight cache.  The summary proposes storing cached activations in
# INT8 or FP8 (section 6, the memory-overhead limitation; section 7, future
# direction 3 "KV cache quantization and memory-efficient DualCache") without
# fixing a scheme.  Reading R13, applied to the LM-head weight (the largest
# per-step read of the path): E4M3 values (OCP FP8: 1 sign, 4 exponent bits
# with bias 7, 3 mantissa bits, subnormals, largest finite 448, no infinity),
# one power-of-two scale per row -- the smallest 2^k with max|row| <= 448 * 2^k
# -- and round to nearest, ties to even.  Hidden rows are quantised the same
# way, per row, at each step (the FP8 tensor-core product takes both operands
# in FP8).  The logits are (s_h s_w) * sum_k qh_k qw_k, evaluated here in float64.
# ---------------------------------------------------------------------------

E4M3_MAX = 448.0


def e4m3_decode(codes):
    """Values of E4M3 byte codes (uint8 array); the two NaN codes (S.1111.111) give NaN."""
    c = np.asarray(codes, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def e4m3_round(y):
    """Nearest E4M3 value to each y (|y| <= 448), ties to the even mantissa.

    The grid step in [2^e, 2^(e+1)) is 2^(e-3) for e >= -6; below 2^-6
    (subnormals) it is 2^-9."""
    y = np.asarray(y, dtype=np.float64)
    assert np.all(np.abs(y) <= E4M3_MAX), "outside the E4M3 range"
    a = np.abs(y)
    out = np.zeros_like(a)
    nz = a > 0
    e = np.floor(np.log2(np.where(nz, a, 1.0)))
    # log2 may land one off at exact powers of two: fix e so that 2^e <= a < 2^(e+1)
    e = np.where(np.exp2(e) > a, e - 1, e)
    e = np.where(np.exp2(e + 1) <= a, e + 1, e)
    step = np.exp2(np.maximum(e, -6.0) - 3.0)
    out = np.where(nz, np.round(a / step) * step, 0.0)      # np.round: half to even, a / step exact
    return np.copysign(out, y)                              # the sign of y, also on zero (IEEE 754 6.3)


def e4m3_encode(v):
    """Byte codes of E4M3 values (exactly representable, finite)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    sign = np.where(np.signbit(v), 0x80, 0)
    codes = np.zeros(v.shape, dtype=np.int64)
    sub = a < 2.0 ** -6
    codes = np.where(sub, np.round(a / 2.0 ** -9), 0).astype(np.int64)
    e = np.floor(np.log2(np.where(sub, 1.0, a)))
    e = np.where(np.exp2(e) > a, e - 1, e)
    e = np.where(np.exp2(e + 1) <= a, e + 1, e)
    m = np.where(sub, 0, a / np.exp2(e) * 8.0 - 8.0)
    normal = ((e + 7).astype(np.int64) << 3) | m.astype(np.int64)
    codes = np.where(sub, codes, normal)
    assert np.array_equal(e4m3_decode(codes | sign), v), "not an E4M3 value"
    return (codes | sign).astype(np.uint8)


def fp8_scale_exponent(amax):
    """Smallest integer k with amax <= 448 * 2^k (0 for amax = 0), decided exactly:
    amax = f 2^x with f in [0.5, 1) (frexp) and 448 = 0.875 * 2^9."""
    if amax == 0:
        return 0
    f, x = math.frexp(float(amax))
    return x - 9 if f <= 0.875 else x - 8


def quantize_fp8_rows(x):
    """Per-row FP8 quantisation of x [R, C] (finite float values): returns (codes uint8 [R, C],
    scales float64 [R] = 2^k); the row's values are codes' values times its scale."""
    x = np.asarray(x, dtype=np.float64)
    codes = np.zeros(x.shape, dtype=np.uint8)
    scales = np.ones(x.shape[0])
    for r in range(x.shape[0]):
        k = fp8_scale_exponent(np.abs(x[r]).max() if x.shape[1] else 0.0)
        scales[r] = 2.0 ** k
        codes[r] = e4m3_encode(e4m3_round(x[r] * 2.0 ** -k))
    return codes, scales


def dequantize_fp8_rows(codes, scales):
    return e4m3_decode(codes) * np.asarray(scales, dtype=np.float64)[:, None]


def lm_head_confidence_fp8(h, w_codes, w_scales):
    """lm_head_confidence with the FP8 weight cache: the hidden rows h [R, H] are quantised
    per row, then both operands are their exact FP8 values times their scales."""
    hq, hs = quantize_fp8_rows(h)
    return lm_head_confidence(dequantize_fp8_rows(hq, hs), dequantize_fp8_rows(w_codes, w_scales))


# ---------------------------------------------------------------------------
# f4: FP8 KV cache -- the summary's own proposal (section 7, future direction 3).
# Reading R14: cached keys and values are stored per (sequence, position, KV
# head) row of d values with the R13 rule (E4M3 codes, one power-of-two scale per
# row); this step's fresh keys and values and the queries stay as they are.  The
# attention over such a cache is the block attention of the dequantised cache.
# ---------------------------------------------------------------------------

def quantize_kv_rows(x):
    """Codes uint8 [b, n, Hkv, d] and scales [b, n, Hkv] of a K or V array [b, n, Hkv, d]."""
    b, n, h, d = x.shape
    codes, scales = quantize_fp8_rows(np.asarray(x, dtype=np.float64).reshape(b * n * h, d))
    return codes.reshape(b, n, h, d), scales.reshape(b, n, h)


def dequantize_kv_rows(codes, scales):
    b, n, h, d = codes.shape
    return dequantize_fp8_rows(codes.reshape(-1, d), scales.reshape(-1)).reshape(b, n, h, d)


def kv_splice_fp8(codes, scales, src, start):
    """The FP8 cache after writing src [b, len, Hkv, d] at positions [start, start + len): the
    window's rows are quantised (R13), every other row is unchanged.  Returns new arrays."""
    qc, qs = quantize_kv_rows(src)
    return kv_splice(codes, qc, start), kv_splice(scales, qs, start)
