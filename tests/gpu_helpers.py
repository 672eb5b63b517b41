"""Shared helpers for the GPU parity tests: device copies of seeded inputs and the
tolerance rules of the parity contract.

Tolerances (decoding method: bf16 inputs, fp32 accumulation):
  * attention output: relative L2 error <= 5e-3 per (sequence, head);
  * confidence: absolute error <= 1e-3; kappa: |d kappa| <= 1e-3 * max(1, |kappa|) + 1e-3;
  * argmax token: bit-exact unless the oracle's top-2 logit gap is < 1e-2;
  * unmask decision: per sequence, the oracle's set, or a set the selection rule gives
    when only exempt comparisons go the other way: a position with |c - tau| < 2e-3
    (threshold), a factor comparison (n + 1)(1 - c_(n)) within (n + 1) 2e-3 of f, or a
    ranking / fallback choice between positions whose kappas are within the kappa
    tolerance (a near tie).  A wrong decision anywhere else fails, whatever its
    neighbours are.
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


def _eps(k):
    """1 - c from the log-odds kappa = log((1 - c) / c)."""
    return 1.0 / (1.0 + math.exp(-k)) if k > -700 else 0.0


def _rank_prefix_ok(kap, masked_idx, sel_idx):
    """`sel_idx` is a most-confident prefix of the masked positions up to near ties of kappa: no
    selected position is less confident than an unselected one by more than the kappa tolerance."""
    rest = [i for i in masked_idx if i not in set(sel_idx)]
    if not sel_idx or not rest:
        return True
    worst_in = max(kap[i] for i in sel_idx)
    best_out = min(kap[i] for i in rest)
    return worst_in <= best_out + kappa_tol(best_out)


def threshold_selection_ok(conf, kap, masked_idx, sel_idx, tau):
    """Can the threshold rule with the progress guarantee (unmask every masked c > tau; if none,
    the single most confident) give `sel_idx`, when only positions with |c - tau| < TAU_EXEMPT may
    fall on either side of tau and the fallback may pick any position tied with the least kappa?

    Positions above the band must be selected and positions below it must not, so the selection is
    either {above} plus some of the band, or -- only if nothing lies above the band -- a single
    fallback pick among the near-tied most confident positions (or a single band position)."""
    above = {i for i in masked_idx if conf[i] - tau >= TAU_EXEMPT}
    band = {i for i in masked_idx if abs(conf[i] - tau) < TAU_EXEMPT}
    sel = set(sel_idx)
    if not masked_idx:
        return not sel
    if sel and above <= sel and sel <= above | band:
        return True
    if not above and len(sel) == 1:
        (j,) = sel
        kmin = min(kap[i] for i in masked_idx)
        return kap[j] <= kmin + kappa_tol(kmin)
    return False


def factor_selection_ok(kap, masked_idx, sel_idx, factor):
    """Can the factor rule (largest n with (n + 1)(1 - c_(n)) < f over the confidence order, at least
    one) give `sel_idx`?  The selection must be a most-confident prefix (near ties of kappa aside), and
    every n between its size and the oracle's count must have (n + 1)(1 - c_(n)) within
    (n + 1) * TAU_EXEMPT of f: only such comparisons may fall on either side of f."""
    if not masked_idx:
        return not sel_idx
    order = sorted(masked_idx, key=lambda i: (kap[i], i))
    vals = [(n + 1) * _eps(kap[order[n - 1]]) for n in range(1, len(order) + 1)]
    n_ref = max([n for n in range(1, len(order) + 1) if vals[n - 1] < factor] + [1])
    n_got = len(sel_idx)
    if n_got < 1 or not _rank_prefix_ok(kap, masked_idx, sel_idx):
        return False
    lo, hi = sorted((n_got, n_ref))
    # n = 1 is never compared (at least one position is unmasked), so the band starts at n = 2
    return all(abs(vals[n - 1] - factor) < (n + 1) * TAU_EXEMPT for n in range(max(lo + 1, 2), hi + 1))


def compare_select(ref: dict, got: dict, tau: float, strategy="threshold", factor: float = 1.0):
    """Compare one step's GPU outputs with the oracle's `decode_step` info.

    Per masked position: confidence within CONF_ATOL, kappa within kappa_tol, argmax token equal
    unless the oracle's top-2 logit gap is below GAP_EXEMPT.  Per sequence, the unmask set must
    equal the oracle's, or be one the selection rule can produce when only the comparisons the
    contract exempts (|c - tau| < TAU_EXEMPT; a factor comparison within the same band; kappa near
    ties in a ranking or fallback) go the other way (threshold_selection_ok, factor_selection_ok,
    _rank_prefix_ok for top-k).

    Returns the number of exempted positions (token differences plus unmask differences); raises
    AssertionError on a mismatch outside the tolerance bands."""
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
        midx = [int(i) for i in np.nonzero(masked[bi])[0]]
        gidx = [int(i) for i in np.nonzero(sel_g)[0]]
        assert set(gidx) <= set(midx), f"sequence {bi}: unmasked a position that was not masked"
        conf, kap = ref["conf"][bi], ref["kappa"][bi]
        if strategy == "threshold":
            ok = threshold_selection_ok(conf, kap, midx, gidx, tau)
        elif strategy == "factor":
            ok = factor_selection_ok(kap, midx, gidx, factor)
        elif strategy == "topk":
            ok = len(gidx) == int(sel_r.sum()) and _rank_prefix_ok(kap, midx, gidx)
        else:
            raise ValueError(strategy)
        if not ok:
            raise AssertionError(f"sequence {bi}: unmask {gidx} vs oracle {list(np.nonzero(sel_r)[0])}")
        exempt += int(np.count_nonzero(sel_g != sel_r))
    return exempt
