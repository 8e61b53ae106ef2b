"""Writes tests/golden/tiny_tokens.json from the oracle alone.

The tiny configuration (2 layers, d_model 128, 4 heads x 32, FFN 512, vocab
512, fp32, weight seed 1001, 32-token prompt) generates 64 tokens in AR,
block diffusion (k = 4 slots per round, 8 rounds) and temperature-0
self-speculation (one drafting forward). Run from the repository root:
    python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle import model  # noqa: E402
from self_speculative_lm_block_b300 import synth  # noqa: E402


def main():
    t = synth.TINY
    cfg = model.Config(layers=t["layers"], d_model=t["d_model"], n_heads=t["n_heads"],
                       n_kv_heads=t["n_kv_heads"], head_dim=t["head_dim"], ffn=t["ffn"],
                       vocab=t["vocab"], dtype="f32", seed=t["seed"])
    w = model.Weights(cfg)
    pr = synth.prompt(t["prompt"], cfg.vocab, cfg.seed)
    out = {"config": "tiny: 2L d128 4x32 ffn512 V512 f32 seed1001 prompt32 gen64",
           "prompt": [int(x) for x in pr]}
    for key, (mode, steps) in {"ar": ("ar", 1), "diff_k4": ("diff", 8),
                               "selfspec_s1": ("selfspec", 1)}.items():
        s = model.Session(cfg, w, max_seq=200)
        s.prefill(pr)
        out[key] = s.generate(mode, t["generate"], steps)
        out[key + "_forwards"] = s.forwards
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_tokens.json"), "w") as f:
        json.dump(out, f, indent=0)


if __name__ == "__main__":
    main()
