"""Large-batch selection workloads for profilers: one warm-up and one
profiled launch each of unmask (top-k, k = 8) and verify/accept over 65536
sequences of 32 slots, the profiled pair inside an NVTX range "select".

    python -m self_speculative_lm_block_b300.profile_select [--batch 65536] [--k 8]
"""
from __future__ import annotations

import argparse

import torch

from . import ndiff as nd
from . import synth


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--batch", type=int, default=65536)
    ap.add_argument("--k", type=int, default=8)
    args = ap.parse_args()
    B, T, k = args.batch, 32, args.k
    conf, pred, mask = synth.unmask_inputs(B, T, 151936, 4001)
    draft, target, _ = synth.draft_target(B, T, 151936, 4002)
    conf, pred, mask, draft, target = (t.cuda() for t in (conf, pred, mask, draft, target))
    z = lambda *shape: torch.zeros(shape, dtype=torch.int32, device="cuda")
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


if __name__ == "__main__":
    main()
