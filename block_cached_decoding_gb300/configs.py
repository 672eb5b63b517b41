"""Workload shapes of the five synthetic settings (sizes and draw parameters only).

The LM-head weight is drawn with standard deviation sqrt(0.05) (tiny setting)
or sqrt(0.02) (LLaDA-8B / Dream-7B shapes): the second argument of N(0, .) is
read as a variance, the only reading under which planted rows give peaked
confidences.  `sigma_w_alt` is the other reading, kept as an all-fallback
stress case.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    prompt_len: int
    gen_length: int
    block_size: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    hidden: int
    vocab: int
    dtype: str               # 'f32' or 'bf16'
    mode: str                # 'dual', 'prefix' or 'none'
    taus: tuple = (0.9,)
    p_plant: float = 0.4
    sigma_w: float = math.sqrt(0.02)
    sigma_w_alt: float = 0.02
    seed: int = 0

    @property
    def seq_len(self) -> int:
        return self.prompt_len + self.gen_length

    @property
    def mask_id(self) -> int:
        return self.vocab          # outside the vocabulary: never predicted

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


TINY = Workload("tiny-fp32", 1, 64, 64, 16, 4, 4, 64, 256, 1024, "f32", "dual",
                taus=(0.9,), p_plant=0.5, sigma_w=math.sqrt(0.05), sigma_w_alt=0.05, seed=100)
LLADA_STEP = Workload("llada8b-prefix-step", 1, 512, 256, 32, 32, 32, 128, 4096, 126464, "bf16", "prefix",
                      taus=(0.9,), seed=101)
LLADA_LOOP = Workload("llada8b-dual-loop-1024", 1, 512, 1024, 32, 32, 32, 128, 4096, 126464, "bf16", "dual",
                      taus=(0.9, 1.0), seed=102)
LLADA_BATCH = Workload("llada8b-dual-batch16", 16, 768, 256, 32, 32, 32, 128, 4096, 126464, "bf16", "dual",
                       taus=(0.7, 0.8, 0.9, 0.95), seed=103)
DREAM = Workload("dream7b-gqa-dual-batch8", 8, 512, 1024, 32, 28, 4, 128, 3584, 152064, "bf16", "dual",
                 taus=(0.9,), seed=104)

ALL = (TINY, LLADA_STEP, LLADA_LOOP, LLADA_BATCH, DREAM)
