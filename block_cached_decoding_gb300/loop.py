"""Block-wise generation loop on the GPU (Algorithm 1 of the Fast-dLLM pages,
section 3.4.4), driving the three ABI calls in lock step over a batch.

The model forward pass is out of scope, so each step's queries, fresh keys and
values and hidden states are drawn by the device twin of the seeded generator
(a stand-in keyed by (sequence, step, position)); caches are re-drawn for each
refresh epoch and written with fdllm_kv_splice(REFRESH) at each block
boundary, standing in for the fused recomputation of every position's K/V
after a block completes.  The refresh epoch is the block index; with
`refresh_interval` r the cache is also refreshed every r steps inside a block
(the refresh-every-r-steps variant the pages report for LLaDA-V), with epoch
block * 1000 + (step in block) // r.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import fdllm as F
from .configs import Workload


def _packed(buf: torch.Tensor, shape) -> torch.Tensor:
    """Dense view of the leading elements of `buf` with `shape` (buffers are sized for the largest step)."""
    n = 1
    for x in shape:
        n *= x
    return buf.view(-1)[:n].view(shape)


@dataclass
class StepResult:
    step: int
    block: int
    block_start: int
    epoch: int                  # refresh epoch of the caches this step read
    unmasked: torch.Tensor      # uint8 [b, B]
    conf: torch.Tensor          # fp32 [b, B]
    kappa: torch.Tensor         # fp32 [b, B]
    argmax: torch.Tensor        # int32 [b, B]
    n_left: torch.Tensor        # int32 [b]
    attn_out: torch.Tensor      # [b, nq, Hq, d]


class BlockDecoder:
    def __init__(self, wl: Workload, *, tau: float = 0.9, strategy: int = F.SELECT_THRESHOLD,
                 factor: float = 1.0, topk: int = 1, sigma_w: float | None = None, device: str = "cuda",
                 refresh_interval: int | None = None, w: torch.Tensor | None = None, fused_update: bool = False):
        """`w`: an LM-head weight already drawn for this workload's (seed, sigma_w, vocab, hidden) to share
        instead of drawing another; `fused_update`: each step's attention also writes the block's fresh K/V
        into the cache window (fdllm_block_attn_update), as a serving loop would."""
        self.wl = wl
        self.refresh_interval = refresh_interval
        self.tau, self.strategy, self.factor, self.topk = tau, strategy, factor, topk
        self.sigma_w = wl.sigma_w if sigma_w is None else sigma_w
        self.dt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
        self.code = F.F32 if wl.dtype == "f32" else F.BF16
        b, n, hq, hkv, d, B = wl.batch, wl.seq_len, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.block_size
        dev = torch.device(device)
        self.fused_update = fused_update
        if w is not None:
            assert w.shape == (wl.vocab, wl.hidden) and w.dtype == self.dt
            self.w = w
        else:
            self.w = torch.empty(wl.vocab, wl.hidden, dtype=self.dt, device=dev)
            F.fdllm_synth_normals(wl.seed, F.SYNTH_W, [], wl.vocab * wl.hidden, 0, self.sigma_w, self.code, self.w)
        self.kc = torch.empty(b, n, hkv, d, dtype=self.dt, device=dev)
        self.vc = torch.empty_like(self.kc)
        self.k_stage = torch.empty_like(self.kc)
        self.v_stage = torch.empty_like(self.kc)
        self.tokens = torch.full((b, n), wl.mask_id, dtype=torch.int32, device=dev)
        prompt = torch.empty(b, wl.prompt_len, dtype=torch.int32, device=dev)
        F.fdllm_synth_prompt(wl.seed, b, wl.prompt_len, wl.vocab, prompt)
        self.tokens.fill_(wl.mask_id)
        self.tokens[:, :wl.prompt_len] = prompt
        nq_max = {"dual": B, "prefix": n - wl.prompt_len, "none": n}[wl.mode]
        self.q = torch.empty(b, nq_max, hq, d, dtype=self.dt, device=dev)
        self.kf = torch.empty(b, nq_max, hkv, d, dtype=self.dt, device=dev)
        self.vf = torch.empty_like(self.kf)
        self.attn_out = torch.empty(b, nq_max, hq, d, dtype=torch.float32, device=dev)
        self.hidden = torch.empty(b, B, wl.hidden, dtype=self.dt, device=dev)
        self.unmasked = torch.empty(b, B, dtype=torch.uint8, device=dev)
        self.conf = torch.empty(b, B, dtype=torch.float32, device=dev)
        self.kappa = torch.empty_like(self.conf)
        self.argmax = torch.empty(b, B, dtype=torch.int32, device=dev)
        self.n_left = torch.empty(b, dtype=torch.int32, device=dev)
        sd = self.select_desc(wl.prompt_len)
        self.sel_ws = torch.empty(F.fdllm_select_workspace_size(sd), dtype=torch.uint8, device=dev)
        self.attn_ws_bytes = max(F.fdllm_attn_workspace_size(self.attn_desc(k))
                                 for k in range(wl.gen_length // B))
        self.attn_ws = torch.empty(max(self.attn_ws_bytes, 16), dtype=torch.uint8, device=dev)

    # -- descriptors -------------------------------------------------------
    def attn_desc(self, k: int) -> F.AttnDesc:
        wl = self.wl
        return F.attn_desc(batch=wl.batch, prompt_len=wl.prompt_len, gen_length=wl.gen_length,
                           block_size=wl.block_size, block_idx=k, n_q_heads=wl.n_q_heads, n_kv_heads=wl.n_kv_heads,
                           head_dim=wl.head_dim, use_cache=0 if wl.mode == "none" else 1,
                           dual_cache=1 if wl.mode == "dual" else 0, dtype=self.code, out_f32=1)

    def select_desc(self, s: int) -> F.SelectDesc:
        wl = self.wl
        return F.select_desc(batch=wl.batch, seq_len=wl.seq_len, block_start=s, block_size=wl.block_size,
                             hidden=wl.hidden, vocab=wl.vocab, mask_id=wl.mask_id, threshold=self.tau,
                             strategy=self.strategy, factor=self.factor, topk=self.topk, dtype=self.code)

    # -- pieces ------------------------------------------------------------
    def query_range(self, k: int) -> tuple[int, int]:
        wl = self.wl
        s = wl.prompt_len + k * wl.block_size
        if wl.mode == "dual":
            return s, s + wl.block_size
        if wl.mode == "prefix":
            return s, wl.seq_len
        return 0, wl.seq_len

    def refresh(self, k: int):
        """Caches recomputed for refresh epoch k (drawn), written by fdllm_kv_splice(REFRESH)."""
        wl = self.wl
        F.fdllm_synth_kv_cache(wl.seed, F.SYNTH_KCACHE, wl.batch, wl.seq_len, wl.n_kv_heads, wl.head_dim, k, 1.0,
                               self.code, self.k_stage)
        F.fdllm_synth_kv_cache(wl.seed, F.SYNTH_VCACHE, wl.batch, wl.seq_len, wl.n_kv_heads, wl.head_dim, k, 1.0,
                               self.code, self.v_stage)
        F.fdllm_kv_splice(F.SPLICE_REFRESH, wl.batch, wl.seq_len, wl.n_kv_heads, wl.head_dim, 0, wl.seq_len,
                          self.code, self.kc, self.vc, self.k_stage, self.v_stage)

    def draw_step_inputs(self, g: int, k: int):
        wl = self.wl
        p0, p1 = self.query_range(k)
        nq = p1 - p0
        b = wl.batch
        F.fdllm_synth_rows(wl.seed, F.SYNTH_Q, b, g, p0, nq, wl.n_q_heads * wl.head_dim, 1.0, self.code, self.q)
        F.fdllm_synth_rows(wl.seed, F.SYNTH_KFRESH, b, g, p0, nq, wl.n_kv_heads * wl.head_dim, 1.0, self.code, self.kf)
        F.fdllm_synth_rows(wl.seed, F.SYNTH_VFRESH, b, g, p0, nq, wl.n_kv_heads * wl.head_dim, 1.0, self.code, self.vf)
        s = wl.prompt_len + k * wl.block_size
        F.fdllm_synth_hidden(wl.seed, b, g, s, wl.block_size, wl.hidden, wl.vocab, wl.p_plant, self.w, self.code,
                             self.hidden)

    def attend(self, desc, q, kf, vf, out, stream=None):
        """The step's block attention (with the cache-window update when the decoder fuses it)."""
        if self.fused_update:
            F.fdllm_block_attn_update(desc, None, q, self.kc, self.vc, kf, vf, out, None, self.attn_ws,
                                      ws_bytes=self.attn_ws_bytes, stream=stream)
        else:
            F.fdllm_block_attn(desc, q, self.kc, self.vc, kf, vf, out, None, self.attn_ws, ws_bytes=self.attn_ws_bytes,
                               stream=stream)

    def reset_tokens(self):
        """Every generated position masked again (the prompt kept): a fresh decode of the same prompt."""
        self.tokens[:, self.wl.prompt_len:] = self.wl.mask_id

    def epoch(self, k: int, n: int) -> int:
        """Refresh epoch of the caches at step n (0-based) of block k."""
        r = self.refresh_interval
        return k if not r else k * 1000 + n // r

    def step(self, g: int, k: int, epoch: int | None = None) -> StepResult:
        """One denoising step of block k: attention over the cache, then confidence select."""
        wl = self.wl
        p0, p1 = self.query_range(k)
        nq = p1 - p0
        self.draw_step_inputs(g, k)
        b, hq, hkv, d = wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
        q, out = _packed(self.q, (b, nq, hq, d)), _packed(self.attn_out, (b, nq, hq, d))
        kf, vf = _packed(self.kf, (b, nq, hkv, d)), _packed(self.vf, (b, nq, hkv, d))
        self.attend(self.attn_desc(k), q, kf, vf, out)
        s = wl.prompt_len + k * wl.block_size
        F.fdllm_confidence_select(self.select_desc(s), self.hidden, self.w, self.tokens, self.unmasked, self.conf,
                                  self.kappa, self.argmax, self.n_left, self.sel_ws)
        return StepResult(g, k, s, self.epoch(k, 0) if epoch is None else epoch, self.unmasked, self.conf, self.kappa,
                          self.argmax, self.n_left, out)

    def capture_blocks(self, max_steps_per_block: int | None = None):
        """One device-driven loop (fdllm_block_loop) per block, captured up front: the step -- inputs drawn at
        the running device step index, the attention and the select -- repeats on the device until the
        block has no mask.  Returns the loops and the device counters (steps per block, running total)."""
        wl = self.wl
        r = self.refresh_interval or 0
        cap = max_steps_per_block or wl.block_size
        nb = wl.gen_length // wl.block_size
        dev = self.w.device
        per_block = torch.zeros(nb, dtype=torch.int64, device=dev)
        total = torch.zeros(1, dtype=torch.int64, device=dev)
        b, hq, hkv, d, B = wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.block_size
        loops = []
        for k in range(nb):
            p0, p1 = self.query_range(k)
            nq = p1 - p0
            s = wl.prompt_len + k * B
            q, out = _packed(self.q, (b, nq, hq, d)), _packed(self.attn_out, (b, nq, hq, d))
            kf, vf = _packed(self.kf, (b, nq, hkv, d)), _packed(self.vf, (b, nq, hkv, d))
            adesc, sdesc = self.attn_desc(k), self.select_desc(s)

            def step(stream, p0=p0, s=s, nq=nq, q=q, out=out, kf=kf, vf=vf, adesc=adesc, sdesc=sdesc):
                F.fdllm_synth_rows_at(wl.seed, F.SYNTH_Q, b, 0, total, p0, nq, hq * d, 1.0, self.code, self.q, stream)
                F.fdllm_synth_rows_at(wl.seed, F.SYNTH_KFRESH, b, 0, total, p0, nq, hkv * d, 1.0, self.code, self.kf,
                                      stream)
                F.fdllm_synth_rows_at(wl.seed, F.SYNTH_VFRESH, b, 0, total, p0, nq, hkv * d, 1.0, self.code, self.vf,
                                      stream)
                F.fdllm_synth_hidden_at(wl.seed, b, 0, total, s, B, wl.hidden, wl.vocab, wl.p_plant, self.w,
                                        self.code, self.hidden, stream)
                self.attend(adesc, q, kf, vf, out, stream)
                F.fdllm_confidence_select(sdesc, self.hidden, self.w, self.tokens, self.unmasked, self.conf,
                                          self.kappa, self.argmax, self.n_left, self.sel_ws, stream=stream)

            def refresh(stream, k=k, counter=per_block[k:k + 1]):
                # the caches of epoch k * 1000 + (step in block) // r, the step read from the loop's counter
                for kind, stage in ((F.SYNTH_KCACHE, self.k_stage), (F.SYNTH_VCACHE, self.v_stage)):
                    F.fdllm_synth_kv_cache_at(wl.seed, kind, wl.batch, wl.seq_len, wl.n_kv_heads, wl.head_dim,
                                              k * 1000, counter, r, 1.0, self.code, stage, stream)
                F.fdllm_kv_splice(F.SPLICE_REFRESH, wl.batch, wl.seq_len, wl.n_kv_heads, wl.head_dim, 0, wl.seq_len,
                                  self.code, self.kc, self.vc, self.k_stage, self.v_stage, stream=stream)

            loops.append(F.BlockLoop(step, self.n_left, b, cap, per_block[k:k + 1], total,
                                     refresh=refresh if r else None, refresh_every=r))
        return loops, per_block, total

    def launch_graph(self, loops):
        """Launch every block's captured loop after its cache refresh, without waiting: returns the device
        counters (steps per block) and the masked count left at the end of each block."""
        graphs, per_block, total = loops
        total.zero_()
        left = torch.zeros(len(graphs), dtype=torch.int32, device=total.device)
        for k, g in enumerate(graphs):
            self.refresh(self.epoch(k, 0))
            g.launch()
            left[k] = self.n_left.max()             # stream-ordered, no host wait
        return per_block, left

    def run_graph(self, max_steps_per_block: int | None = None, loops=None):
        """The same decode as `run` with every block a device-driven loop (`capture_blocks`, or the given
        capture): the host only launches each block's loop after its cache refresh and reads the step
        counts once at the end.  Returns (tokens, steps per block)."""
        wl = self.wl
        cap = max_steps_per_block or wl.block_size
        own = loops is None
        if own:
            loops = self.capture_blocks(max_steps_per_block)
        graphs = loops[0]
        per_block, left = self.launch_graph(loops)
        steps = per_block.tolist()                  # one synchronisation for the whole decode
        left = left.tolist()
        if own:
            for g in graphs:
                g.close()
        for k, n_left in enumerate(left):
            if n_left:
                raise RuntimeError(f"block {k} did not finish within {cap} steps")
        return self.tokens, steps

    # -- per-sequence blocks (each sequence moves on as soon as its own block is decoded) --------------
    def _ragged_state(self):
        """Device state of a per-sequence generation, reset to every sequence at its first block with
        its caches refreshed for it (refresh epoch = the sequence's block index)."""
        wl = self.wl
        if wl.mode != "dual":
            raise ValueError("per-sequence blocks need DualCache")
        b, dev = wl.batch, self.w.device
        if not hasattr(self, "rg"):
            self.rg = {"n_blocks": wl.gen_length // wl.block_size, "block_size": wl.block_size,
                       "block_idx": torch.zeros(b, dtype=torch.int32, device=dev),
                       "block_start": torch.zeros(b, dtype=torch.int32, device=dev),
                       "seq_steps": torch.zeros(b, dtype=torch.int32, device=dev),
                       "refresh_flags": torch.zeros(b, dtype=torch.uint8, device=dev),
                       "done": torch.zeros(b, dtype=torch.uint8, device=dev)}
        rg = self.rg
        rg["block_idx"].zero_()
        rg["block_start"].fill_(wl.prompt_len)
        rg["seq_steps"].zero_()
        rg["refresh_flags"].zero_()
        rg["done"].zero_()
        self.reset_tokens()
        self.ragged_refresh(None, only=None)
        return rg

    def ragged_refresh(self, stream, only="flags"):
        """The caches of the flagged sequences (all with only=None) recomputed for their current block:
        the synthetic stand-in draws refresh epoch block_idx[b] straight into the caches."""
        wl, rg = self.wl, self.rg
        flags = rg["refresh_flags"] if only == "flags" else None
        for kind, cache in ((F.SYNTH_KCACHE, self.kc), (F.SYNTH_VCACHE, self.vc)):
            F.fdllm_synth_kv_cache_seq(wl.seed, kind, wl.batch, wl.seq_len, wl.n_kv_heads, wl.head_dim,
                                       rg["block_idx"], flags, 1.0, self.code, cache, stream)

    def ragged_step(self, stream=None):
        """One step of every sequence at its own block: inputs drawn at the sequence's own step and
        window, attention with the window update, select (the *_ragged calls)."""
        wl, rg = self.wl, self.rg
        b, hq, hkv, d, B = wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.block_size
        q, out = _packed(self.q, (b, B, hq, d)), _packed(self.attn_out, (b, B, hq, d))
        kf, vf = _packed(self.kf, (b, B, hkv, d)), _packed(self.vf, (b, B, hkv, d))
        st, p0 = rg["seq_steps"], rg["block_start"]
        F.fdllm_synth_rows_seq(wl.seed, F.SYNTH_Q, b, st, p0, B, hq * d, 1.0, self.code, q, stream)
        F.fdllm_synth_rows_seq(wl.seed, F.SYNTH_KFRESH, b, st, p0, B, hkv * d, 1.0, self.code, kf, stream)
        F.fdllm_synth_rows_seq(wl.seed, F.SYNTH_VFRESH, b, st, p0, B, hkv * d, 1.0, self.code, vf, stream)
        F.fdllm_synth_hidden_seq(wl.seed, b, st, p0, B, wl.hidden, wl.vocab, wl.p_plant, self.w, self.code,
                                 self.hidden, stream)
        F.fdllm_block_attn_update(self.attn_desc(0), rg["block_idx"], q, self.kc, self.vc, kf, vf, out, None,
                                  self.attn_ws, ws_bytes=self.attn_ws_bytes, stream=stream)
        F.fdllm_confidence_select_ragged(self.select_desc(wl.prompt_len), p0, self.hidden, self.w, self.tokens,
                                         self.unmasked, self.conf, self.kappa, self.argmax, self.n_left,
                                         self.sel_ws, stream=stream)
        return out

    def run_ragged(self, hook=None):
        """Host-driven per-sequence generation: after each step the host reads the masked counts and moves
        each finished block's sequence on (as fdllm_block_loop_create_ragged's control kernel does), then
        refreshes the moved sequences' caches.  `hook(decoder, out, blocks, starts, steps, done)` sees
        each step's outputs and the state it ran with.  Returns (tokens, steps per sequence)."""
        wl = self.wl
        rg = self._ragged_state()
        nb, B = rg["n_blocks"], wl.block_size
        blk = [0] * wl.batch
        steps = [0] * wl.batch
        done = [False] * wl.batch
        for _ in range(nb * B):
            if all(done):
                break
            out = self.ragged_step()
            left = self.n_left.cpu().tolist()
            if hook is not None:
                hook(self, out, list(blk), [wl.prompt_len + k * B for k in blk], list(steps), list(done))
            flags = [0] * wl.batch
            for i in range(wl.batch):
                if done[i]:
                    continue
                steps[i] += 1
                if left[i] == 0:
                    if blk[i] + 1 == nb:
                        done[i] = True
                    else:
                        blk[i] += 1
                        flags[i] = 1
            rg["block_idx"].copy_(torch.tensor(blk, dtype=torch.int32))
            rg["block_start"].copy_(torch.tensor([wl.prompt_len + k * B for k in blk], dtype=torch.int32))
            rg["seq_steps"].copy_(torch.tensor(steps, dtype=torch.int32))
            rg["refresh_flags"].copy_(torch.tensor(flags, dtype=torch.uint8))
            if any(flags):
                self.ragged_refresh(None)
        if not all(done):
            raise RuntimeError("a sequence did not finish within n_blocks * block_size steps")
        return self.tokens, steps

    def capture_ragged(self):
        """The per-sequence generation captured as one device-driven loop (fdllm_block_loop_create_ragged);
        returns (loop, device step counter)."""
        wl = self.wl
        rg = self._ragged_state()
        counter = torch.zeros(1, dtype=torch.int64, device=self.w.device)
        loop = F.BlockLoop(lambda stream: self.ragged_step(stream), self.n_left, wl.batch,
                           rg["n_blocks"] * wl.block_size, counter, refresh=lambda stream: self.ragged_refresh(stream),
                           ragged=rg)
        return loop, counter

    def launch_ragged(self, loop):
        """A fresh generation through a captured per-sequence loop: state, tokens and caches reset on the
        device, then the loop launched; nothing waits on the host."""
        self._ragged_state()
        loop.launch()

    def run_ragged_graph(self):
        """The same generation as `run_ragged` as one device-driven loop: the host launches it once and reads
        the per-sequence step counts at the end."""
        loop, _ = self.capture_ragged()
        try:
            self.launch_ragged(loop)
            steps = self.rg["seq_steps"].tolist()
            done = self.rg["done"].tolist()
        finally:
            loop.close()
        if not all(done):
            raise RuntimeError("a sequence did not finish within n_blocks * block_size steps")
        return self.tokens, steps

    def run(self, hook=None, max_steps_per_block: int | None = None):
        """Decode every block left to right; returns (tokens, steps per block)."""
        wl = self.wl
        steps = []
        g = 0
        cap = max_steps_per_block or wl.block_size
        for k in range(wl.gen_length // wl.block_size):
            n = 0
            ep = self.epoch(k, 0)
            self.refresh(ep)
            while True:
                if n > 0 and self.epoch(k, n) != ep:
                    ep = self.epoch(k, n)
                    self.refresh(ep)
                r = self.step(g, k, ep)
                if hook is not None:
                    hook(self, r)
                g += 1
                n += 1
                if int(r.n_left.max().item()) == 0:
                    break
                if n >= cap:
                    raise RuntimeError(f"block {k} did not finish within {cap} steps")
            steps.append(n)
        return self.tokens, steps
