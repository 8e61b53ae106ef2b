"""Projection workloads for profilers: one launch each of the wide projection
kernel (a batch of token rows) and of the fused LM head with its argmax
epilogue, inside an NVTX range named "proj" after an untimed warm-up call.

    python -m self_speculative_lm_block_b300.profile_gemm [--rows 2048] [--n 6144] [--k 4096]
        [--lm-rows 32] [--vocab 151936]

Defaults: the QKV projection of the 8B-shaped model for 64 sequences x 32
tokens (2048 x 6144 x 4096, 66 MB of operands), and the 8B LM head
(151936 x 4096 bf16, 1.24 GB) for one 32-token block.
"""
from __future__ import annotations

import argparse

import torch

from . import ndiff as nd


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--rows", type=int, default=2048)
    ap.add_argument("--n", type=int, default=6144)
    ap.add_argument("--k", type=int, default=4096)
    ap.add_argument("--lm-rows", type=int, default=32)
    ap.add_argument("--vocab", type=int, default=151936)
    args = ap.parse_args()
    gen = torch.Generator(device="cuda").manual_seed(7)
    x = torch.randn((args.rows, args.k), device="cuda", generator=gen).to(torch.bfloat16)
    w = (torch.randn((args.n, args.k), device="cuda", generator=gen) * 0.02).to(torch.bfloat16)
    xl = torch.randn((args.lm_rows, args.k), device="cuda", generator=gen).to(torch.bfloat16)
    wl = (torch.randn((args.vocab, args.k), device="cuda", generator=gen) * 0.02).to(torch.bfloat16)
    nd.gemm_bf16(x, w)
    nd.lm_head_argmax(xl, wl, args.vocab - 1)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("proj")
    nd.gemm_bf16(x, w)
    nd.lm_head_argmax(xl, wl, args.vocab - 1)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    nd.ndiff_check()


if __name__ == "__main__":
    main()
