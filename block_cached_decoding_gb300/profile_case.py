"""Run one hot-path call on a chosen shape a few times (the command ncu profiles).

    python -m block_cached_decoding_gb300.profile_case select --vocab 32768 --reps 3
    python -m block_cached_decoding_gb300.profile_case select --fp8w --reps 3
    python -m block_cached_decoding_gb300.profile_case select --f32 --vocab 32768 --hidden 1024 --reps 3
    python -m block_cached_decoding_gb300.profile_case attn --mode prefix --reps 3
    python -m block_cached_decoding_gb300.profile_case attn --mode prefix --update --reps 3
    python -m block_cached_decoding_gb300.profile_case splice --reps 3

Inputs come from the device twin of the seeded generator; shapes default to
the LLaDA-8B single-step workload (block 0, 32 masked rows, 32 heads x 128).
"""
from __future__ import annotations

import argparse

import torch

from . import configs
from . import fdllm as F


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("op", choices=["select", "attn", "splice"])
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--prompt", type=int, default=512)
    ap.add_argument("--gen", type=int, default=256)
    ap.add_argument("--block", type=int, default=32)
    ap.add_argument("--block-idx", type=int, default=0)
    ap.add_argument("--hidden", type=int, default=4096)
    ap.add_argument("--vocab", type=int, default=126464)
    ap.add_argument("--hq", type=int, default=32)
    ap.add_argument("--hkv", type=int, default=32)
    ap.add_argument("--d", type=int, default=128)
    ap.add_argument("--mode", default="prefix", choices=["dual", "prefix", "none"])
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--fp8w", action="store_true", help="select through the FP8 weight cache")
    ap.add_argument("--f32", action="store_true",
                    help="fp32 hidden rows and weight (the CUDA-core LM head, then select_kernel)")
    ap.add_argument("--fp8kv", action="store_true", help="attention over the FP8 KV cache")
    ap.add_argument("--update", action="store_true",
                    help="attention with the cache-window update (fdllm_block_attn_update)")
    ap.add_argument("--ragged", action="store_true",
                    help="per-sequence blocks: sequence i at block i mod (gen / block) (DualCache attention, select)")
    ap.add_argument("--time", action="store_true", help="report the mean call time over the reps (CUDA events)")
    a = ap.parse_args()
    wl = configs.LLADA_STEP
    dev = torch.device("cuda", 0)
    b, n, B = a.batch, a.prompt + a.gen, a.block
    s = a.prompt + a.block_idx * B
    code = F.BF16
    if a.op == "select":
        if a.f32:
            code = F.F32
        tdt = torch.float32 if a.f32 else torch.bfloat16
        W = torch.empty(a.vocab, a.hidden, dtype=tdt, device=dev)
        F.fdllm_synth_normals(wl.seed, F.SYNTH_W, [], a.vocab * a.hidden, 0, wl.sigma_w, code, W)
        hid = torch.empty(b, B, a.hidden, dtype=tdt, device=dev)
        F.fdllm_synth_hidden(wl.seed, b, 0, s, B, a.hidden, a.vocab, wl.p_plant, W, code, hid)
        tokens0 = torch.full((b, n), a.vocab, dtype=torch.int32, device=dev)
        tokens = tokens0.clone()
        d = F.select_desc(batch=b, seq_len=n, block_start=s, block_size=B, hidden=a.hidden, vocab=a.vocab,
                          mask_id=a.vocab, threshold=0.9, dtype=code)
        outs = [torch.empty(b, B, dtype=t, device=dev) for t in (torch.uint8, torch.float32, torch.float32, torch.int32)]
        nleft = torch.empty(b, dtype=torch.int32, device=dev)
        starts = torch.tensor([a.prompt + (i % (a.gen // B)) * B for i in range(b)], dtype=torch.int32, device=dev)
        if a.ragged:
            ws = torch.empty(F.fdllm_select_workspace_size(d), dtype=torch.uint8, device=dev)
            def call():
                tokens.copy_(tokens0)
                F.fdllm_confidence_select_ragged(d, starts, hid, W, tokens, *outs, nleft, ws)
        elif a.fp8w:
            wq = torch.empty(a.vocab, a.hidden, dtype=torch.uint8, device=dev)
            wsc = torch.empty(a.vocab, dtype=torch.float32, device=dev)
            F.fdllm_quantize_fp8_rows(a.vocab, a.hidden, code, W, wq, wsc)
            del W
            ws = torch.empty(F.fdllm_select_fp8w_workspace_size(d), dtype=torch.uint8, device=dev)
            def call():
                tokens.copy_(tokens0)
                F.fdllm_confidence_select_fp8w(d, hid, wq, wsc, tokens, *outs, nleft, ws)
        else:
            ws = torch.empty(F.fdllm_select_workspace_size(d), dtype=torch.uint8, device=dev)
            def call():
                tokens.copy_(tokens0)
                F.fdllm_confidence_select(d, hid, W, tokens, *outs, nleft, ws)
    elif a.op == "attn":
        d = F.attn_desc(batch=b, prompt_len=a.prompt, gen_length=a.gen, block_size=B, block_idx=a.block_idx,
                        n_q_heads=a.hq, n_kv_heads=a.hkv, head_dim=a.d, use_cache=0 if a.mode == "none" else 1,
                        dual_cache=1 if a.mode == "dual" else 0, dtype=code, out_f32=0)
        nq = F.fdllm_attn_query_count(d)
        p0 = {"dual": s, "prefix": s, "none": 0}[a.mode]
        kc = torch.empty(b, n, a.hkv, a.d, dtype=torch.bfloat16, device=dev)
        vc = torch.empty_like(kc)
        F.fdllm_synth_kv_cache(wl.seed, F.SYNTH_KCACHE, b, n, a.hkv, a.d, 0, 1.0, code, kc)
        F.fdllm_synth_kv_cache(wl.seed, F.SYNTH_VCACHE, b, n, a.hkv, a.d, 0, 1.0, code, vc)
        q = torch.empty(b, nq, a.hq, a.d, dtype=torch.bfloat16, device=dev)
        kf = torch.empty(b, nq, a.hkv, a.d, dtype=torch.bfloat16, device=dev)
        vf = torch.empty_like(kf)
        F.fdllm_synth_rows(wl.seed, F.SYNTH_Q, b, 0, p0, nq, a.hq * a.d, 1.0, code, q)
        F.fdllm_synth_rows(wl.seed, F.SYNTH_KFRESH, b, 0, p0, nq, a.hkv * a.d, 1.0, code, kf)
        F.fdllm_synth_rows(wl.seed, F.SYNTH_VFRESH, b, 0, p0, nq, a.hkv * a.d, 1.0, code, vf)
        out = torch.empty(b, nq, a.hq, a.d, dtype=torch.bfloat16, device=dev)
        wsb = F.fdllm_attn_workspace_size(d)
        ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
        blocks = torch.tensor([i % (a.gen // B) for i in range(b)], dtype=torch.int32, device=dev)
        if a.fp8kv:
            kq = torch.empty(b, n, a.hkv, a.d, dtype=torch.uint8, device=dev)
            vq = torch.empty_like(kq)
            ksc = torch.empty(b, n, a.hkv, dtype=torch.float32, device=dev)
            vsc = torch.empty_like(ksc)
            F.fdllm_kv_splice_fp8(F.SPLICE_REFRESH, b, n, a.hkv, a.d, 0, n, code, kq, ksc, vq, vsc, kc, vc)
            del kc, vc
        def call():
            if a.fp8kv:
                F.fdllm_block_attn_fp8kv(d, blocks if a.ragged else None, q, kq, ksc, vq, vsc, kf, vf, out, None, ws,
                                         ws_bytes=wsb)
            elif a.update:
                F.fdllm_block_attn_update(d, blocks if a.ragged else None, q, kc, vc, kf, vf, out, None, ws,
                                          ws_bytes=wsb)
            elif a.ragged:
                F.fdllm_block_attn_ragged(d, blocks, q, kc, vc, kf, vf, out, None, ws, ws_bytes=wsb)
            else:
                F.fdllm_block_attn(d, q, kc, vc, kf, vf, out, None, ws, ws_bytes=wsb)
    else:
        kc = torch.zeros(b, n, a.hkv, a.d, dtype=torch.bfloat16, device=dev)
        vc = torch.zeros_like(kc)
        ks = torch.ones(b, n, a.hkv, a.d, dtype=torch.bfloat16, device=dev)
        vs = torch.ones_like(ks)
        def call():
            F.fdllm_kv_splice(F.SPLICE_REFRESH, b, n, a.hkv, a.d, 0, n, code, kc, vc, ks, vs)
    if a.time:
        for _ in range(3):
            call()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(a.reps):
            call()
        e1.record()
        torch.cuda.synchronize()
        print(f"{a.op} {vars(a)}: {e0.elapsed_time(e1) / a.reps * 1e3:.2f} us per call (mean of {a.reps}, L2 warm)")
    else:
        for _ in range(a.reps):
            call()
    torch.cuda.synchronize()
    st, detail = F.fdllm_last_device_error()
    if st != F.OK:
        raise SystemExit(f"device error word set: site {detail}")
    print(f"{a.op}: {a.reps} calls ok")


if __name__ == "__main__":
    main()
