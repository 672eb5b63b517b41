"""Seeded synthetic inputs shared by the CUDA path, the oracle and the benchmarks.

This module holds random-number generation only; none of the decoding method's
arithmetic lives here.  Every value is a pure function of (seed, tensor kind, a
few integer coordinates, element index), so the CPU side (this file, numpy) and
the device side (``csrc/synth.cu``) produce the *same bytes* without sharing
code.  Both implement the same published generator:

* SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): the i-th output of a stream with state ``s`` is
  ``fmix(s + (i + 1) * GAMMA)`` with the 64-bit finaliser ``fmix`` below.
* Normal deviates by the Irwin-Hall construction ("sum of twelve uniforms minus
  six"): twelve 16-bit uniforms ``u_j = (k_j + 1/2) / 2^16`` taken from three
  SplitMix64 outputs.  ``sum(u_j) - 6 = (sum(k_j) - 393210) / 65536`` is an
  integer over a power of two, so it is exact in float32 on both sides.
  Mean 0, variance 1 - 2^-32, support [-6, 6].
* Scaling by sigma is one float32 multiply (round to nearest even), and the
  conversion to bfloat16 is round-to-nearest-even on the float32 bits.  The
  device side uses ``__fmul_rn`` / ``__fadd_rn`` so no FMA contraction changes
  a rounding.

Tensor kinds and their coordinates (one stream per coordinate tuple):

============  =======================  =========================================
kind          coordinates              element index
============  =======================  =========================================
W      (1)    ()                       v * H + k          (LM-head weight [V, H])
KCACHE (2)    (b, epoch)               (n * Hkv + h) * d + j
VCACHE (3)    (b, epoch)               (n * Hkv + h) * d + j
Q      (4)    (b, step, pos)           h * d + j          (Hq heads)
KFRESH (5)    (b, step, pos)           h * d + j          (Hkv heads)
VFRESH (6)    (b, step, pos)           h * d + j
HID    (7)    (b, step, pos)           k                  (hidden state row)
PLANT  (8)    (b, step, pos)           output 0: plant draw, output 1: target
PROMPT (9)    (b,)                     n                  (prompt token ids)
============  =======================  =========================================

A hidden-state row is ``z + 6 * W[t]`` (float32 add of the float32 product)
with probability ``p_plant``, else ``z``; ``t`` is uniform over the vocabulary.
The planted direction makes the softmax over the vocabulary peaked at ``t``.
"""
from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

KIND_W, KIND_KCACHE, KIND_VCACHE, KIND_Q, KIND_KFRESH, KIND_VFRESH, KIND_HID, KIND_PLANT, KIND_PROMPT = range(1, 10)


def _fmix(z):
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = z ^ (z >> np.uint64(30))
        z = z * _M1
        z = z ^ (z >> np.uint64(27))
        z = z * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def splitmix(state, i):
    """i-th SplitMix64 output of the stream whose state is ``state`` (vectorised over i)."""
    i = np.asarray(i, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _fmix(np.uint64(state) + (i + np.uint64(1)) * GAMMA)


def stream_key(seed: int, *coords: int) -> np.uint64:
    """Chain the coordinates into one 64-bit stream state: s <- splitmix(s, c)."""
    s = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
    for c in coords:
        s = np.uint64(splitmix(s, np.uint64(int(c) & 0xFFFFFFFFFFFFFFFF)))
    return s


def normal12_f32(key: np.uint64, n: int, offset: int = 0) -> np.ndarray:
    """float32 Irwin-Hall-12 normals for element indices offset .. offset+n-1.

    Element i uses SplitMix64 outputs 3i, 3i+1, 3i+2 of the stream; each output
    contributes its four 16-bit fields as integer uniforms k_j."""
    idx = np.arange(offset, offset + n, dtype=np.uint64) * np.uint64(3)
    lanes = np.uint64(0x0000FFFF0000FFFF)
    acc = np.zeros(n, dtype=np.uint64)
    for part in range(3):
        r = splitmix(key, idx + np.uint64(part))
        acc += (r & lanes) + ((r >> np.uint64(16)) & lanes)   # two 32-bit lanes of partial sums
    tot = (acc & np.uint64(0xFFFFFFFF)) + (acc >> np.uint64(32))
    return ((tot.astype(np.int64) - 393210).astype(np.float32) / np.float32(65536.0)).astype(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def scaled_normals(key, n, sigma: float, dtype: str, offset: int = 0) -> np.ndarray:
    """sigma * z in float32, then stored as `dtype` ('f32' -> float32, 'bf16' -> uint16 bits)."""
    z = normal12_f32(key, n, offset)
    v = (z * np.float32(sigma)).astype(np.float32)
    return v if dtype == "f32" else f32_to_bf16_bits(v)


def as_f32(a: np.ndarray, dtype: str) -> np.ndarray:
    """Stored values (float32 or bf16 bit patterns) as float32."""
    return a if dtype == "f32" else bf16_bits_to_f32(a)


# ---------------------------------------------------------------------------
# whole tensors
# ---------------------------------------------------------------------------

def lm_head_weight(seed, vocab, hidden, sigma_w, dtype):
    """W [V, H]."""
    return scaled_normals(stream_key(seed, KIND_W), vocab * hidden, sigma_w, dtype).reshape(vocab, hidden)


def kv_cache(seed, kind, batch, seq_len, n_kv, head_dim, epoch, dtype, sigma=1.0):
    """K or V cache [b, N, Hkv, d] drawn for refresh epoch `epoch` (kind KCACHE or VCACHE)."""
    per = seq_len * n_kv * head_dim
    out = [scaled_normals(stream_key(seed, kind, b, epoch), per, sigma, dtype) for b in range(batch)]
    return np.stack(out).reshape(batch, seq_len, n_kv, head_dim)


def per_position(seed, kind, batch, step, positions, width, dtype, sigma=1.0):
    """Rows drawn per (b, step, pos): returns [b, len(positions), width]."""
    out = np.empty((batch, len(positions), width), dtype=np.float32 if dtype == "f32" else np.uint16)
    for b in range(batch):
        for i, p in enumerate(positions):
            out[b, i] = scaled_normals(stream_key(seed, kind, b, step, p), width, sigma, dtype)
    return out


def plant_draws(seed, batch, step, positions, p_plant, vocab):
    """(planted bool [b, n], target int64 [b, n]) for each (b, step, pos)."""
    thr = np.uint64(int(np.floor(p_plant * (1 << 24))))
    planted = np.zeros((batch, len(positions)), dtype=bool)
    target = np.zeros((batch, len(positions)), dtype=np.int64)
    for b in range(batch):
        for i, p in enumerate(positions):
            k = stream_key(seed, KIND_PLANT, b, step, p)
            r0 = splitmix(k, 0)
            r1 = splitmix(k, 1)
            planted[b, i] = (r0 >> np.uint64(40)) < thr
            target[b, i] = int(((r1 >> np.uint64(32)) * np.uint64(vocab)) >> np.uint64(32))
    return planted, target


def lm_head_row(seed, v, hidden, sigma_w, dtype):
    """Row v of W without drawing the rest of W."""
    return scaled_normals(stream_key(seed, KIND_W), hidden, sigma_w, dtype, offset=v * hidden)


def hidden_states(seed, batch, step, positions, hidden, vocab, sigma_w, dtype, p_plant):
    """Hidden rows [b, n, H]: z + 6 * W[t] (float32 ops) when planted, else z; then stored dtype.

    Returns (rows, planted [b, n], target [b, n])."""
    planted, target = plant_draws(seed, batch, step, positions, p_plant, vocab)
    out = np.empty((batch, len(positions), hidden), dtype=np.float32 if dtype == "f32" else np.uint16)
    for b in range(batch):
        for i, p in enumerate(positions):
            z = normal12_f32(stream_key(seed, KIND_HID, b, step, p), hidden)
            if planted[b, i]:
                w = as_f32(lm_head_row(seed, int(target[b, i]), hidden, sigma_w, dtype), dtype)
                z = (z + (np.float32(6.0) * w).astype(np.float32)).astype(np.float32)
            out[b, i] = z if dtype == "f32" else f32_to_bf16_bits(z)
    return out, planted, target


def prompt_tokens(seed, batch, prompt_len, vocab):
    """Prompt ids [b, P], uniform over [0, V)."""
    out = np.empty((batch, prompt_len), dtype=np.int32)
    for b in range(batch):
        r = splitmix(stream_key(seed, KIND_PROMPT, b), np.arange(prompt_len, dtype=np.uint64))
        out[b] = (((r >> np.uint64(32)) * np.uint64(vocab)) >> np.uint64(32)).astype(np.int32)
    return out
