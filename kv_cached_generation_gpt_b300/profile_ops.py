"""Launch one library kernel a few times at a workload's shapes (for ncu captures).

    python -m kv_cached_generation_gpt_b300.profile_ops attn_decode [--batch 64] [--t 768] [--launches 4]
    python -m kv_cached_generation_gpt_b300.profile_ops gemm --m 32768 --n 2304 --k 768 [--block-n 256]
    python -m kv_cached_generation_gpt_b300.profile_ops attn_prefill [--batch 64] [--t 512]
    python -m kv_cached_generation_gpt_b300.profile_ops sample [--batch 64] [--top-k 50]
    python -m kv_cached_generation_gpt_b300.profile_ops linear_decode --m 64 --n 2304 --k 768 [--gemm-splits 4]

Shapes default to GPT-2 124M (12 heads of 64, vocab 50304, block 1024).  Inputs are seeded
random tensors; every launch goes through the C ABI and the op status is checked at the end.
"""
from __future__ import annotations

import argparse

import torch

from kv_cached_generation_gpt_b300 import gpt as G


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("op", choices=["attn_decode", "attn_prefill", "gemm", "linear_decode", "sample"])
    ap.add_argument("--batch", type=int, default=64)
    ap.add_argument("--heads", type=int, default=12)
    ap.add_argument("--block", type=int, default=1024)
    ap.add_argument("--t", type=int, default=768, help="cached keys (decode) or prompt length (prefill)")
    ap.add_argument("--splits", type=int, default=1)
    ap.add_argument("--m", type=int, default=64)
    ap.add_argument("--n", type=int, default=2304)
    ap.add_argument("--k", type=int, default=768)
    ap.add_argument("--block-n", type=int, default=0)
    ap.add_argument("--gemm-splits", type=int, default=1)
    ap.add_argument("--hilo", action="store_true")
    ap.add_argument("--vocab", type=int, default=50304)
    ap.add_argument("--top-k", type=int, default=50)
    ap.add_argument("--launches", type=int, default=4)
    a = ap.parse_args()
    torch.manual_seed(0)
    dev = torch.device("cuda", 0)
    B, nh, hs = a.batch, a.heads, 64
    if a.op == "attn_decode":
        kc = torch.randn(B, nh, a.block, hs, device=dev).to(torch.bfloat16)
        vc = torch.randn(B, nh, a.block, hs, device=dev).to(torch.bfloat16)
        q = torch.randn(B, nh, 1, hs, device=dev).to(torch.bfloat16)
        y = torch.empty(B, nh * hs, device=dev, dtype=torch.bfloat16)
        lo = torch.empty_like(y)
        pos = torch.tensor([a.t - 1], dtype=torch.int32, device=dev)
        run = lambda: G.gpt_attention_decode(q, kc, vc, pos, a.splits, y, lo)
    elif a.op == "attn_prefill":
        kc = torch.randn(B, nh, a.block, hs, device=dev).to(torch.bfloat16)
        vc = torch.randn(B, nh, a.block, hs, device=dev).to(torch.bfloat16)
        q = torch.randn(B, nh, a.t, hs, device=dev).to(torch.bfloat16)
        y = torch.empty(B * a.t, nh * hs, device=dev, dtype=torch.bfloat16)
        run = lambda: G.gpt_attention_prefill(q, kc, vc, 0, y)
    elif a.op == "gemm":
        rows = 2 * a.m if a.hilo else a.m
        A = torch.randn(rows, a.k, device=dev).to(torch.bfloat16)
        W = (0.02 * torch.randn(a.n, a.k, device=dev)).to(torch.bfloat16)
        out = torch.empty(a.m, a.n, device=dev)
        run = lambda: G.gpt_linear_bf16(A, W, None, out, a.m, hilo=a.hilo, block_n=a.block_n, splits=a.gemm_splits)
    elif a.op == "linear_decode":
        A = torch.randn(2 * a.m, a.k, device=dev).to(torch.bfloat16)
        W = (0.02 * torch.randn(a.n, a.k, device=dev)).to(torch.bfloat16)
        out = torch.empty(a.m, a.n, device=dev)
        run = lambda: G.gpt_linear_decode_bf16(A, W, None, out, a.m, splits=a.gemm_splits)
    else:
        logits = torch.randn(B, a.vocab, device=dev)
        tok = torch.empty(B, dtype=torch.int32, device=dev)
        run = lambda: G.gpt_sample(logits, 1.0, a.top_k, 7, 0, tok)
    for _ in range(a.launches):
        run()
    torch.cuda.synchronize()
    status = G.gpt_op_status()
    if status != G.GPT_OK:
        raise SystemExit(f"op status {status}: {G.lib().gpt_strerror(status).decode()}")
    print(f"{a.op}: {a.launches} launches ok")


if __name__ == "__main__":
    main()
