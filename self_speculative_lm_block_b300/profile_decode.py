"""Decode-cycle workload for profilers: builds a random-init model, prefills a
prompt, then runs one AR step and one self-speculation cycle inside an NVTX
range named "decode", so that a profiler can be limited to those launches
(`--nvtx --nvtx-include "decode/"`).

    python -m self_speculative_lm_block_b300.profile_decode [--layers 36] [--vocab 151936]
        [--prompt 1024] [--steps 1] [--batch 1]

The default is the 8B-shaped model (d_model 4096, 32/8 heads x 128, SwiGLU 12288,
bf16); --layers 1 --vocab 4096 keeps one layer's projections at full width with
a device footprint near 0.5 GB. --batch B decodes B sequences together (the
prompts then have ragged lengths in [prompt/2, prompt]) through the batch calls.
"""
from __future__ import annotations

import argparse

import torch

from . import ndiff as nd
from . import synth


def main():
    ap = argparse.ArgumentParser()
    c = synth.MODEL_8B
    ap.add_argument("--layers", type=int, default=c["layers"])
    ap.add_argument("--vocab", type=int, default=c["vocab"])
    ap.add_argument("--prompt", type=int, default=c["prompt"])
    ap.add_argument("--steps", type=int, default=1, help="drafting forwards per block")
    ap.add_argument("--batch", type=int, default=1)
    args = ap.parse_args()
    m = nd.Model(args.layers, c["d_model"], c["n_heads"], c["n_kv_heads"], c["head_dim"], c["ffn"],
                 args.vocab, dtype="bf16", max_seq=args.prompt + 256, seed=c["seed"],
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
        m.step(nd.NDIFF_MODE_SELFSPEC, args.steps)
    else:
        m.step_batch(nd.NDIFF_MODE_AR)
        m.step_batch(nd.NDIFF_MODE_SELFSPEC, args.steps)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    m.close()
    print("ok")


if __name__ == "__main__":
    main()
