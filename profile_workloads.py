#!/usr/bin/env python3
"""Workloads for profilers (ncu): each runs a few launches of one part of the
decode step inside an NVTX range, so that a capture can be limited to them
(`--nvtx --nvtx-include "<range>/"`). Nothing here is timed or checked; the
benchmark is bench.py and the parity tests are under tests/.

    python profile_workloads.py decode [--layers 36] [--vocab 151936] [--prompt 1024]
                                       [--steps 1] [--batch 1]
        range "decode": one AR step and one self-speculation cycle of the
        8B-shaped random-init model (d_model 4096, 32/8 heads x 128, SwiGLU
        12288, bf16), after a prefill. --layers 1 --vocab 4096 keeps one
        layer's projections at full width with a device footprint near 0.5 GB;
        --batch B decodes B sequences together (ragged prompts in
        [prompt/2, prompt]) through the batch calls; --quad runs a quadratic
        self-speculation cycle (candidates 0 and 1) instead of the linear one.

    python profile_workloads.py gemm [--rows 2048] [--n 6144] [--k 4096]
                                     [--lm-rows 32] [--vocab 151936]
        range "proj": one launch each of the wide projection kernel (default:
        the QKV projection of 64 sequences x 32 tokens) and of the fused LM head
        with its argmax epilogue (default: the 8B LM head for one block), after
        an untimed warm-up call of each.

    python profile_workloads.py select [--batch 65536] [--k 8]
        range "select": one unmask (top-k) and one verify/accept launch over
        65536 sequences of 32 slots, after a warm-up pair.

    python profile_workloads.py attn [--workload single|batched|long] [--reps 2]
        range "attn": block attention (CAUSAL, 32/8 heads x 128, 32-token
        block) on the seeded inputs of a configuration (single: batch 1 x 4096
        keys; batched: 64 sequences, prefixes in [512, 8192]; long: batch 4 x
        32768), --reps launches after three warm-up launches.
"""
from __future__ import annotations

import argparse
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

from self_speculative_lm_block_b300 import ndiff as nd  # noqa: E402
from self_speculative_lm_block_b300 import synth  # noqa: E402


def decode(args):
    c = synth.MODEL_8B
    m = nd.Model(args.layers, c["d_model"], c["n_heads"], c["n_kv_heads"], c["head_dim"], c["ffn"],
                 args.vocab, dtype="bf16", max_seq=args.prompt + 512, seed=c["seed"],
                 batch=args.batch)
    if args.batch == 1:
        m.prefill(synth.prompt(args.prompt, args.vocab, c["seed"]))
    else:
        lens = [args.prompt // 2 + (i * 37) % (args.prompt // 2 + 1) for i in range(args.batch)]
        m.prefill_batch([list(synth.prompt(n, args.vocab, c["seed"] + i)) for i, n in enumerate(lens)])
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("decode")
    if args.batch == 1:
        m.step(nd.NDIFF_MODE_AR)
        if args.quad:
            m.step(nd.NDIFF_MODE_SELFSPEC_QUAD, cands=(0, 1))
        else:
            m.step(nd.NDIFF_MODE_SELFSPEC, args.steps)
    else:
        m.step_batch(nd.NDIFF_MODE_AR)
        m.step_batch(nd.NDIFF_MODE_SELFSPEC, args.steps)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    m.close()


def gemm(args):
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


def select(args):
    B, T, k = args.batch, 32, args.k
    conf, pred, mask = synth.unmask_inputs(B, T, 151936, 4001)
    draft, target, _ = synth.draft_target(B, T, 151936, 4002)
    conf, pred, mask, draft, target = (t.cuda() for t in (conf, pred, mask, draft, target))

    def z(*shape):
        return torch.zeros(shape, dtype=torch.int32, device="cuda")

    blk, dr, ch, mk = z(B, T), z(B, T), z(B, k), mask.clone()
    L, n, com, kv = z(B), z(B), z(B, T), z(B)
    for rng in (False, True):
        mk.copy_(mask)
        torch.cuda.synchronize()
        if rng:
            torch.cuda.nvtx.range_push("select")
        nd.ndiff_unmask(conf, pred, B, T, k, mk, blk, dr, ch)
        nd.ndiff_verify_accept(draft, target, B, T, L, com, n, kv)
        if rng:
            torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
    nd.ndiff_check()


def attn(args):
    c = {"single": synth.ATTN_SINGLE, "batched": synth.ATTN_BATCHED, "long": synth.ATTN_LONG}[args.workload]
    lengths = synth.attn_lengths(c["B"], c["seed"], c["P_lo"], c["P_hi"])
    Lmax = int(c["P_hi"]) + c["T"]
    inp = synth.attn_inputs(c["B"], c["T"], c["Hq"], c["Hkv"], c["D"], lengths, Lmax, c["seed"])
    q, k, v, kv = inp.q.cuda(), inp.k_cache.cuda(), inp.v_cache.cuda(), inp.kv_len.cuda()
    for _ in range(3):
        nd.block_attn(q, k, v, kv, nd.NDIFF_CAUSAL, inp.scale)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("attn")
    for _ in range(args.reps):
        nd.block_attn(q, k, v, kv, nd.NDIFF_CAUSAL, inp.scale)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    nd.ndiff_check()


def main():
    ap = argparse.ArgumentParser()
    sub = ap.add_subparsers(dest="what", required=True)
    c = synth.MODEL_8B
    d = sub.add_parser("decode")
    d.add_argument("--layers", type=int, default=c["layers"])
    d.add_argument("--vocab", type=int, default=c["vocab"])
    d.add_argument("--prompt", type=int, default=c["prompt"])
    d.add_argument("--steps", type=int, default=1, help="drafting forwards per block")
    d.add_argument("--batch", type=int, default=1)
    d.add_argument("--quad", action="store_true", help="a quadratic self-speculation cycle")
    g = sub.add_parser("gemm")
    g.add_argument("--rows", type=int, default=2048)
    g.add_argument("--n", type=int, default=6144)
    g.add_argument("--k", type=int, default=4096)
    g.add_argument("--lm-rows", type=int, default=32)
    g.add_argument("--vocab", type=int, default=151936)
    s = sub.add_parser("select")
    s.add_argument("--batch", type=int, default=65536)
    s.add_argument("--k", type=int, default=8)
    a = sub.add_parser("attn")
    a.add_argument("--workload", default="single", choices=["single", "batched", "long"])
    a.add_argument("--reps", type=int, default=2)
    args = ap.parse_args()
    {"decode": decode, "gemm": gemm, "select": select, "attn": attn}[args.what](args)
    print("ok")


if __name__ == "__main__":
    main()
