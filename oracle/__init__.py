"""Oracle: a plain, slow, float64 CPU statement of what the decode step computes.

TEST INFRASTRUCTURE ONLY. Only the tests, the package entry's smoke() check and
the benchmark's CPU-baseline leg may import this package. The CUDA product path
never calls it, and it imports nothing from the CUDA path; the two share only
the seeded input generators (which hold none of the method's arithmetic).

Modules:
  attention   block-causal GQA attention (plain definition)
  decode      logits reduction, diffusion unmask step, verify/accept
  philox      Philox4x64-10 and the Box-Muller weight stream
  numerics    bf16 round-to-nearest-even
  model       the random-init tri-mode model and its AR / DIFF / SELFSPEC loops

Parity pins (what fixes each part independently of the oracle itself) live in
tests/test_oracle_*.py. Parity unpinned: the readings that only a trained
checkpoint could confirm (the logit shift convention, the commit forward of a
diffusion block, the number of drafting forwards, the RoPE pairing) — they are
checked for internal consistency only.
"""
