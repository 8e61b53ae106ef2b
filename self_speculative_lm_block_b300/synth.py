"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module only draws random numbers and lays them out; it holds none of the
decode-step arithmetic. Every tensor comes from NumPy's PCG64 seeded through a
SeedSequence of (seed, tag, index...), so any single sequence or row can be
regenerated on its own (the oracle checks sampled rows of full-size inputs that
way). bf16 tensors are drawn as float32 and rounded to bf16 with torch's
round-to-nearest-even conversion.

Workload shapes follow the 8B-like configurations: 32 query heads / 8 KV heads
of dimension 128, a 32-token query block, KV prefixes of 4096 (single), uniform
in [512, 8192] (batched) or 32768 (long context), and a 151936-entry vocabulary.
"""
from __future__ import annotations

import dataclasses
import numpy as np
import torch

BLOCK = 32

# Tags keep the streams of different tensors apart.
_TAG_Q, _TAG_K, _TAG_V, _TAG_LEN, _TAG_LOGITS = 1, 2, 3, 4, 5
_TAG_DRAFT, _TAG_TARGET, _TAG_CONF, _TAG_MASK, _TAG_PRED, _TAG_PROMPT = 6, 7, 8, 9, 10, 11


def _rng(*words: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(w) for w in words])))


def normal_bf16(shape, sigma: float, *seed_words: int) -> torch.Tensor:
    """float32 N(0, sigma^2) draws rounded to bf16 (CPU tensor)."""
    a = _rng(*seed_words).standard_normal(size=shape, dtype=np.float32)
    if sigma != 1.0:
        a *= np.float32(sigma)
    return torch.from_numpy(a).to(torch.bfloat16)


def normal_f32(shape, sigma: float, *seed_words: int) -> torch.Tensor:
    a = _rng(*seed_words).standard_normal(size=shape, dtype=np.float32)
    if sigma != 1.0:
        a *= np.float32(sigma)
    return torch.from_numpy(a)


# --------------------------------------------------------------------------
# Attention inputs
# --------------------------------------------------------------------------
@dataclasses.dataclass
class AttnInputs:
    q: torch.Tensor        # [B][T][Hq][D]
    k_cache: torch.Tensor  # [B][Hkv][Lmax][D]
    v_cache: torch.Tensor  # [B][Hkv][Lmax][D]
    kv_len: torch.Tensor   # [B] int32 (committed prefix P_b)
    T: int
    scale: float


def attn_lengths(B: int, seed: int, lo: int, hi: int) -> np.ndarray:
    """Prefix lengths P_b uniform on the integers [lo, hi] (lo == hi: fixed)."""
    if lo == hi:
        return np.full(B, lo, dtype=np.int32)
    return _rng(seed, _TAG_LEN).integers(lo, hi + 1, size=B, dtype=np.int64).astype(np.int32)


def attn_sequence(seed: int, b: int, Hq: int, Hkv: int, D: int, T: int, P: int, dtype):
    """One sequence's q [T][Hq][D] and its valid cache rows k, v [Hkv][P+T][D]."""
    mk = normal_bf16 if dtype == torch.bfloat16 else normal_f32
    q = mk((T, Hq, D), 1.0, seed, _TAG_Q, b)
    k = mk((Hkv, P + T, D), 1.0, seed, _TAG_K, b)
    v = mk((Hkv, P + T, D), 1.0, seed, _TAG_V, b)
    return q, k, v


def attn_inputs(B: int, T: int, Hq: int, Hkv: int, D: int, lengths, Lmax: int, seed: int,
                dtype=torch.bfloat16, fill_tail: float = 0.0) -> AttnInputs:
    """Q ~ N(0,1), K/V ~ N(0,1) in the cache rows [0, P_b+T); the rows beyond
    are set to `fill_tail` (NaN checks that they are never read)."""
    lengths = np.asarray(lengths, dtype=np.int32)
    q = torch.empty((B, T, Hq, D), dtype=dtype)
    kc = torch.full((B, Hkv, Lmax, D), fill_tail, dtype=dtype)
    vc = torch.full((B, Hkv, Lmax, D), fill_tail, dtype=dtype)
    for b in range(B):
        P = int(lengths[b])
        assert P + T <= Lmax
        qb, kb, vb = attn_sequence(seed, b, Hq, Hkv, D, T, P, dtype)
        q[b] = qb
        kc[b, :, : P + T] = kb
        vc[b, :, : P + T] = vb
    return AttnInputs(q, kc, vc, torch.from_numpy(lengths.copy()), T, 1.0 / float(np.sqrt(D)))


# --------------------------------------------------------------------------
# Logits / verification / unmask inputs
# --------------------------------------------------------------------------
def logits_row(seed: int, r: int, V: int, sigma: float, dtype=torch.bfloat16) -> torch.Tensor:
    mk = normal_bf16 if dtype == torch.bfloat16 else normal_f32
    return mk((V,), sigma, seed, _TAG_LOGITS, r)


def logits(R: int, V: int, sigma: float, seed: int, dtype=torch.bfloat16, ld: int | None = None):
    """[R][ld] logits; row r ~ N(0, sigma^2) from its own stream. Columns
    [V, ld) are padding holding a value that would win every argmax if read."""
    ld = V if ld is None else ld
    out = torch.empty((R, ld), dtype=dtype)
    if ld > V:
        out[:, V:] = 1e4  # padding that would win every argmax if it were read
    for r in range(R):
        out[r, :V] = logits_row(seed, r, V, sigma, dtype)
    return out


def draft_target(B: int, T: int, V: int, seed: int):
    """(draft, target) int32 [B][T]: target uniform ids; draft equals target
    before a first-mismatch slot m_b ~ U{0..T} (m_b == T: full match) and is
    drawn independently (never equal at m_b) from there on."""
    rng = _rng(seed, _TAG_TARGET)
    target = rng.integers(0, V, size=(B, T), dtype=np.int64)
    m = rng.integers(0, T + 1, size=B)
    draft = target.copy()
    rd = _rng(seed, _TAG_DRAFT)
    for b in range(B):
        if m[b] < T:
            draft[b, m[b]] = (target[b, m[b]] + 1 + rd.integers(0, V - 1)) % V
            draft[b, m[b] + 1:] = rd.integers(0, V, size=T - m[b] - 1)
    return (torch.from_numpy(draft.astype(np.int32)), torch.from_numpy(target.astype(np.int32)),
            m.astype(np.int32))


def unmask_inputs(B: int, T: int, V: int, seed: int, ties: bool = False, all_masked: bool = False):
    """conf float32 [B][T] ~ U(0,1] (ties=True: multiples of 1/16), pred ids
    [B][T], mask bits [B] ~ Bernoulli(1/2) per slot (or all set)."""
    rng = _rng(seed, _TAG_CONF)
    if ties:
        conf = (rng.integers(1, 17, size=(B, T)) / 16.0).astype(np.float32)
    else:
        conf = (1.0 - rng.random(size=(B, T), dtype=np.float32)).astype(np.float32)
    pred = _rng(seed, _TAG_PRED).integers(0, V, size=(B, T), dtype=np.int64).astype(np.int32)
    full = (1 << T) - 1
    if all_masked:
        mask = np.full(B, full, dtype=np.uint64)
    else:
        bits = _rng(seed, _TAG_MASK).integers(0, 2, size=(B, T))
        mask = (bits * (1 << np.arange(T, dtype=np.uint64))).sum(axis=1).astype(np.uint64)
    return (torch.from_numpy(conf), torch.from_numpy(pred),
            torch.from_numpy(mask.astype(np.uint32).view(np.int32)))


def prompt(n: int, vocab: int, seed: int) -> np.ndarray:
    """n token ids uniform on [0, vocab-1): the last id (the [MASK] id) is never drawn."""
    return _rng(seed, _TAG_PROMPT).integers(0, vocab - 1, size=n, dtype=np.int64).astype(np.int32)


# --------------------------------------------------------------------------
# The five workload configurations
# --------------------------------------------------------------------------
TINY = dict(layers=2, d_model=128, n_heads=4, n_kv_heads=4, head_dim=32, ffn=512, vocab=512,
            dtype="f32", prompt=32, generate=64, seed=1001)
ATTN_SINGLE = dict(B=1, Hq=32, Hkv=8, D=128, T=BLOCK, P_lo=4096, P_hi=4096, seed=1002)
ATTN_BATCHED = dict(B=64, Hq=32, Hkv=8, D=128, T=BLOCK, P_lo=512, P_hi=8192, seed=1003,
                    V=151936, logit_sigma=4.0)
ATTN_LONG = dict(B=4, Hq=32, Hkv=8, D=128, T=BLOCK, P_lo=32768, P_hi=32768, seed=1004)
MODEL_8B = dict(layers=36, d_model=4096, n_heads=32, n_kv_heads=8, head_dim=128, ffn=12288,
                vocab=151936, dtype="bf16", prompt=1024, generate=512, seed=1005)
