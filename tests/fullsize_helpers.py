"""Host-side inputs for the full-size parity tests: the whole LM-head weight drawn
by the numpy generator on all host cores (a spawn pool, so no CUDA state is
forked), cached per (seed, V, H, sigma) for the test session."""
from __future__ import annotations

import multiprocessing as mp
import os
from multiprocessing import shared_memory

import numpy as np

from block_cached_decoding_gb300 import synth

_CACHE = {}


def _fill(args):
    name, shape, v0, v1, seed, sigma, dtype = args
    shm = shared_memory.SharedMemory(name=name)
    w = np.ndarray(shape, dtype=np.float32, buffer=shm.buf)
    h = shape[1]
    raw = synth.scaled_normals(synth.stream_key(seed, synth.KIND_W), (v1 - v0) * h, sigma, dtype, offset=v0 * h)
    w[v0:v1] = synth.as_f32(raw, dtype).reshape(v1 - v0, h)
    del w
    shm.close()
    return v1 - v0


def weight_f64(seed: int, vocab: int, hidden: int, sigma: float, dtype: str = "bf16") -> np.ndarray:
    """W [V, H] as float64 (the stored bf16 values, exactly)."""
    key = (seed, vocab, hidden, round(sigma, 9), dtype)
    if key in _CACHE:
        return _CACHE[key]
    _CACHE.clear()                       # keep at most one full weight in memory
    shape = (vocab, hidden)
    shm = shared_memory.SharedMemory(create=True, size=vocab * hidden * 4)
    try:
        jobs = [(shm.name, shape, v, min(v + 2048, vocab), seed, sigma, dtype) for v in range(0, vocab, 2048)]
        with mp.get_context("spawn").Pool(os.cpu_count() or 1) as pool:
            assert sum(pool.map(_fill, jobs)) == vocab
        w = np.ndarray(shape, dtype=np.float32, buffer=shm.buf).astype(np.float64)
    finally:
        shm.close()
        shm.unlink()
    _CACHE[key] = w
    return w
