"""Shared helpers for the GPU parity tests: device copies of seeded inputs and the
tolerance rules of the parity contract.

Tolerances (decoding method: bf16 inputs, fp32 accumulation):
  * attention output: relative L2 error <= 5e-3 per (sequence, head);
  * confidence: absolute error <= 1e-3; kappa: |d kappa| <= 1e-3 * max(1, |kappa|) + 1e-3;
  * argmax token: bit-exact unless the oracle's top-2 logit gap is < 1e-2;
  * unmask decision: bit-exact unless |c - tau| < 2e-3 at that position, or the step
    fell back to one position and the two candidates' kappas are within the kappa
    tolerance (a near tie).
"""
from __future__ import annotations

import math

import numpy as np
import torch

from block_cached_decoding_gb300 import fdllm as F
from block_cached_decoding_gb300 import synth
from oracle import fdllm_oracle as O

ATTN_RTOL = 5e-3
CONF_ATOL = 1e-3
GAP_EXEMPT = 1e-2
TAU_EXEMPT = 2e-3


def ensure_built():
    import os
    if not os.path.exists(F.LIB_PATH):
        from block_cached_decoding_gb300 import build
        build.build()
    F.lib()


def dev(arr: np.ndarray, dtype: str) -> torch.Tensor:
    """Stored values (float32, or bf16 bit patterns as uint16) to a CUDA tensor."""
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(arr)).cuda()
    return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).cuda().view(torch.bfloat16)


def f64(arr: np.ndarray, dtype: str) -> np.ndarray:
    return synth.as_f32(arr, dtype).astype(np.float64)


def tdtype(dtype: str):
    return torch.float32 if dtype == "f32" else torch.bfloat16


def code(dtype: str) -> int:
    return F.F32 if dtype == "f32" else F.BF16


def rel_l2(a: np.ndarray, b: np.ndarray) -> float:
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def assert_attention_close(o_gpu: np.ndarray, o_ref: np.ndarray, tol=ATTN_RTOL):
    b, nq, hq, d = o_ref.shape
    worst = 0.0
    for bi in range(b):
        for h in range(hq):
            e = rel_l2(o_gpu[bi, :, h], o_ref[bi, :, h])
            worst = max(worst, e)
            assert e <= tol, f"relative L2 {e:.3e} > {tol} at batch {bi} head {h}"
    return worst


class SelectOutputs:
    """Device buffers for one fdllm_confidence_select call."""

    def __init__(self, desc, batch, block_size):
        self.unmasked = torch.zeros(batch, block_size, dtype=torch.uint8, device="cuda")
        self.conf = torch.zeros(batch, block_size, dtype=torch.float32, device="cuda")
        self.kappa = torch.zeros(batch, block_size, dtype=torch.float32, device="cuda")
        self.argmax = torch.zeros(batch, block_size, dtype=torch.int32, device="cuda")
        self.n_left = torch.zeros(batch, dtype=torch.int32, device="cuda")
        self.ws = torch.empty(F.fdllm_select_workspace_size(desc), dtype=torch.uint8, device="cuda")

    def run(self, desc, hidden, w, tokens):
        F.fdllm_confidence_select(desc, hidden, w, tokens, self.unmasked, self.conf, self.kappa, self.argmax,
                                  self.n_left, self.ws)

    def host(self):
        torch.cuda.synchronize()
        return {"unmask": self.unmasked.cpu().numpy().astype(bool), "conf": self.conf.cpu().numpy(),
                "kappa": self.kappa.cpu().numpy(), "token": self.argmax.cpu().numpy(),
                "n_left": self.n_left.cpu().numpy()}


def kappa_tol(k):
    return 1e-3 * max(1.0, abs(k)) + 1e-3


def compare_select(ref: dict, got: dict, tau: float, strategy="threshold", factor: float = 1.0):
    """Compare one step's GPU outputs with the oracle's `decode_step` info.

    Returns the number of exempted positions; raises AssertionError on a mismatch
    outside the tolerance bands."""
    masked = ref["masked_before"]
    b, B = masked.shape
    exempt = 0
    for bi in range(b):
        for i in range(B):
            if not masked[bi, i]:
                assert math.isnan(got["conf"][bi, i]) and got["token"][bi, i] == -1 and not got["unmask"][bi, i]
                continue
            c_ref, k_ref = ref["conf"][bi, i], ref["kappa"][bi, i]
            assert abs(got["conf"][bi, i] - c_ref) <= CONF_ATOL, (bi, i, got["conf"][bi, i], c_ref)
            assert abs(got["kappa"][bi, i] - k_ref) <= kappa_tol(k_ref), (bi, i, got["kappa"][bi, i], k_ref)
            if got["token"][bi, i] != ref["token"][bi, i]:
                assert ref["gap"][bi, i] < GAP_EXEMPT, (bi, i, got["token"][bi, i], ref["token"][bi, i], ref["gap"][bi, i])
                exempt += 1
        sel_g, sel_r = got["unmask"][bi], ref["unmask"][bi]
        if np.array_equal(sel_g, sel_r):
            continue
        diff = np.nonzero(sel_g != sel_r)[0]
        near_tau = [i for i in diff if abs(ref["conf"][bi, i] - tau) < TAU_EXEMPT]
        if strategy == "threshold" and len(near_tau) == len(diff):
            exempt += len(diff)
            continue
        # a fallback (or rank-based) pick between near-tied candidates
        if sel_g.sum() == sel_r.sum():
            kg = sorted(ref["kappa"][bi, np.nonzero(sel_g)[0]])
            kr = sorted(ref["kappa"][bi, np.nonzero(sel_r)[0]])
            if all(abs(x - y) <= kappa_tol(y) for x, y in zip(kg, kr)):
                exempt += len(diff)
                continue
        if strategy == "threshold":
            # near-threshold flips change whether the step falls back; accept when the only
            # disagreement is explained by positions within the tau band
            if any(abs(ref["conf"][bi, i] - tau) < TAU_EXEMPT for i in np.nonzero(masked[bi])[0]):
                exempt += len(diff)
                continue
        if strategy == "factor":
            # the rule compares (n + 1) (1 - c_(n)) with f; a value within the confidence
            # tolerance of f may fall on either side
            eps = np.sort(1.0 - ref["conf"][bi, np.nonzero(masked[bi])[0]])
            if any(abs((n + 2) * e - factor) < (n + 2) * TAU_EXEMPT for n, e in enumerate(eps)):
                exempt += len(diff)
                continue
        raise AssertionError(f"sequence {bi}: unmask {np.nonzero(sel_g)[0]} vs oracle {np.nonzero(sel_r)[0]}")
    return exempt
