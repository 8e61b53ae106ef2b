"""The random-init tri-mode model and its three decode modes, float64, step by step.

Sources (page title, section):
- "Nemotron-Labs-Diffusion: A Tri-Mode Language Model Unifying Autoregressive,
  Diffusion, and Self-Speculation Decoding" (hotpaper.ai), Abstract: one model,
  three decoding modes; in self-speculation diffusion drafts and AR verifies.
- "NVIDIA 发布 Nemotron-Labs Diffusion 语言模型系列" (fintech-frontier-insights),
  "三种生成模式": one checkpoint switched between AR (token by token, left to
  right), diffusion (a 32-token block refined over several denoising rounds)
  and self-speculation (diffusion drafts, AR verifies; at temperature 0 the
  output equals pure AR output).
- "Nemotron-Labs-Diffusion: 一种统一自回归、扩散和自推测解码的三模式语言模型"
  (ai-feeds.com), "方法": masked-token denoising objective, shared backbone, no
  extra parameters for the attention pattern.
- gsyq.cn explainer, §2.3 "自推测解码": accept the agreeing prefix, replace the
  first mismatch with the verifier's token.

Readings where the pages are silent (each is listed in the design notes):
- Logits of input slot i predict the token after it, in every mode (one LM
  head serves all modes). Block input = [last, x1..x31] at positions
  n-1 .. n+30; output slot i predicts the token at position n+i.
- [MASK] id = vocab-1; prompts never contain it; it is excluded from argmax.
- DIFF: `steps` BIDIR forwards, each unmasking k = 32/steps slots, then one
  BIDIR forward of [last, d0..d30] that writes the block's KV (counted).
- SELFSPEC: the same drafting forwards, then one CAUSAL forward of
  [last, d0..d30]; accept the longest agreeing prefix plus the correction.
- Fused self-speculation ("NVIDIA 发布 Nemotron-Labs Diffusion 语言模型系列"
  (fintech-frontier-insights), 吞吐量数据: linear and quadratic
  self-speculation; the linear one is read as one forward that verifies a
  block and drafts the next): a forward of [last, d0..d30] (CAUSAL) followed
  by [d31, MASK x 31] at the next 32 positions (BIDIR, over the prefix plus
  the block under verification). The agreeing prefix plus the correction is
  committed; when all 32 drafts were accepted, the second half's argmaxes are
  the next block's draft, otherwise the next cycle drafts afresh (one BIDIR
  forward). Each fused forward counts as one forward.
- Quadratic self-speculation (same page and table: 6.4x against linear 6x)
  is read as drafting the next block, in the verifying forward, for more than
  the one acceptance length the linear variant assumes: for L = 32 as above,
  and for each candidate length L < 32 in a given set, a block of 32 [MASK]
  inputs at positions P+L+1 .. P+L+32 over the prefix plus the verified
  block's first L+1 inputs (the state after committing L drafts and the
  correction; the correction itself is not known inside the forward, so its
  slot stays masked). If the verified L is 32 or a candidate, that block's
  argmaxes are the next draft, else the next cycle drafts afresh. The whole
  forward counts as one.
- Threshold sampler (either mode): BIDIR drafting rounds until no slot is
  masked, each fixing the masked slots whose confidence reaches tau (else the
  most confident one) after revising earlier slots (oracle.decode.
  unmask_threshold); tau and tau_revise are compared in float32, the
  precision the confidences come in.
- Architecture: pre-norm, RMSNorm with unit gain and eps, rotate-half RoPE
  (pairs (i, i+D/2), base 10000, absolute positions), SwiGLU FFN, untied LM
  head, all weights N(0, 0.02^2) from the Philox stream of oracle.philox.
- bf16 model: weights bf16; the inputs of every matrix product (normed
  activations, attention output, SwiGLU output) and q/k/v after RoPE are
  rounded to bf16; the residual stream and all sums stay wide. f32 model: no
  rounding (the oracle computes in float64 throughout).

Every row of a forward is computed independently of the other rows (per-row
matrix-vector products), so a CAUSAL forward of T tokens gives the same rows as
T single-token forwards: self-speculation reproduces AR exactly here.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import attention, decode, philox
from .numerics import round_f32_to_bf16, round_to_bf16

BLOCK = 32


@dataclasses.dataclass
class Config:
    layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    dtype: str = "f32"          # "f32" | "bf16"
    rope_base: float = 10000.0
    eps: float = 1e-6
    seed: int = 0

    @property
    def mask_id(self) -> int:
        return self.vocab - 1


# tensor ids of the weight stream
def tid_embed() -> int:
    return 0


def tid_layer(l: int, j: int) -> int:
    """j: 0 q, 1 k, 2 v, 3 o, 4 gate, 5 up, 6 down."""
    return 1 + 8 * l + j


def tid_lm(cfg: Config) -> int:
    return 1 + 8 * cfg.layers


def tensor_shape(cfg: Config, tid: int):
    d, D = cfg.d_model, cfg.head_dim
    if tid == 0 or tid == tid_lm(cfg):
        return (cfg.vocab, d)
    j = (tid - 1) % 8
    return {0: (cfg.n_heads * D, d), 1: (cfg.n_kv_heads * D, d), 2: (cfg.n_kv_heads * D, d),
            3: (d, cfg.n_heads * D), 4: (cfg.ffn, d), 5: (cfg.ffn, d), 6: (d, cfg.ffn)}[j]


class Weights:
    """Weights drawn on demand from the Philox stream (float64 values)."""

    def __init__(self, cfg: Config):
        self.cfg = cfg
        self._cache: dict[int, np.ndarray] = {}

    def _values(self, tid: int, start: int, count: int) -> np.ndarray:
        w = philox.weight_values(self.cfg.seed, tid, start, count)   # float32
        if self.cfg.dtype == "bf16":
            return round_f32_to_bf16(w)       # exact float32 input: one nearest-even rounding
        return w.astype(np.float64)

    def full(self, tid: int) -> np.ndarray:
        if tid not in self._cache:
            shape = tensor_shape(self.cfg, tid)
            self._cache[tid] = self._values(tid, 0, shape[0] * shape[1]).reshape(shape)
        return self._cache[tid]

    def rows(self, tid: int, rows) -> np.ndarray:
        shape = tensor_shape(self.cfg, tid)
        if tid in self._cache:
            return self._cache[tid][np.asarray(rows)]
        return np.stack([self._values(tid, int(r) * shape[1], shape[1]) for r in rows])

    def drop(self, tid: int) -> None:
        self._cache.pop(tid, None)


def rmsnorm(x: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps), unit gain, per row."""
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def rope(x: np.ndarray, pos: np.ndarray, base: float) -> np.ndarray:
    """Rotate-half RoPE. x [T][H][D], pos [T] absolute positions."""
    D = x.shape[-1]
    half = D // 2
    inv = base ** (-(2.0 * np.arange(half)) / D)              # [half]
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv[None, :]  # [T][half]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def rowwise_matmul(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """y[t] = W x[t] for each row separately (so a row never depends on T)."""
    return np.stack([w @ x[t] for t in range(x.shape[0])])


class Session:
    """KV cache + decode state of one sequence (batch 1)."""

    def __init__(self, cfg: Config, weights: Weights | None = None, max_seq: int = 4096):
        self.cfg = cfg
        self.w = weights or Weights(cfg)
        D = cfg.head_dim
        self.k = [np.zeros((cfg.n_kv_heads, max_seq, D)) for _ in range(cfg.layers)]
        self.v = [np.zeros((cfg.n_kv_heads, max_seq, D)) for _ in range(cfg.layers)]
        self.kv_len = 0
        self.last = -1
        self.tokens: list[int] = []
        self.forwards = 0
        self.accept_lens: list[int] = []
        self.revisions = 0
        self.rounds = 0
        self.pending_draft = None

    def _rb(self, x: np.ndarray) -> np.ndarray:
        return round_to_bf16(x) if self.cfg.dtype == "bf16" else x

    def forward(self, ids, mode: int, vocab_rows=None) -> np.ndarray:
        """One forward of block tokens `ids` at positions kv_len .. kv_len+T-1.
        Writes their K/V into the cache at those positions (scratch beyond the
        committed prefix) and returns logits [T][V] (or [T][len(vocab_rows)])."""
        cfg, w = self.cfg, self.w
        ids = np.asarray(ids, dtype=np.int64)
        T = ids.shape[0]
        P = self.kv_len
        D, Hq, Hkv = cfg.head_dim, cfg.n_heads, cfg.n_kv_heads
        pos = np.arange(P, P + T)
        x = w.rows(tid_embed(), ids)                                 # [T][d]
        for l in range(cfg.layers):
            h = self._rb(rmsnorm(x, cfg.eps))
            q = rowwise_matmul(h, w.full(tid_layer(l, 0))).reshape(T, Hq, D)
            k = rowwise_matmul(h, w.full(tid_layer(l, 1))).reshape(T, Hkv, D)
            v = rowwise_matmul(h, w.full(tid_layer(l, 2))).reshape(T, Hkv, D)
            q = self._rb(rope(q, pos, cfg.rope_base))
            k = self._rb(rope(k, pos, cfg.rope_base))
            v = self._rb(v)
            self.k[l][:, P:P + T] = k.transpose(1, 0, 2)
            self.v[l][:, P:P + T] = v.transpose(1, 0, 2)
            o = attention.block_attn(q[None], self.k[l][None], self.v[l][None], [P], mode,
                                     1.0 / np.sqrt(D))[0]            # [T][Hq][D]
            o = self._rb(o).reshape(T, Hq * D)
            x = x + rowwise_matmul(o, w.full(tid_layer(l, 3)))
            h = self._rb(rmsnorm(x, cfg.eps))
            g = rowwise_matmul(h, w.full(tid_layer(l, 4)))
            u = rowwise_matmul(h, w.full(tid_layer(l, 5)))
            a = self._rb(silu(g) * u)
            x = x + rowwise_matmul(a, w.full(tid_layer(l, 6)))
        h = self._rb(rmsnorm(x, cfg.eps))
        wl = w.full(tid_lm(cfg)) if vocab_rows is None else w.rows(tid_lm(cfg), vocab_rows)
        self.forwards += 1
        return rowwise_matmul(h, wl)

    # ---- session ---------------------------------------------------------
    def prefill(self, prompt) -> None:
        prompt = [int(t) for t in prompt]
        self.kv_len = 0
        self.tokens = []
        if len(prompt) > 1:
            self.forward(prompt[:-1], attention.CAUSAL)
        self.forwards = 0
        self.kv_len = len(prompt) - 1
        self.last = prompt[-1]
        self.pending_draft = None

    def _argmax(self, logits):
        return decode.logits_reduce(logits, exclude_id=self.cfg.mask_id)

    def step_ar(self) -> list[int]:
        logits = self.forward([self.last], attention.CAUSAL)
        a = int(self._argmax(logits)[0][0])
        self.kv_len += 1
        self.last = a
        self.tokens.append(a)
        return [a]

    def draft(self, steps: int) -> np.ndarray:
        assert BLOCK % steps == 0
        k = BLOCK // steps
        block_in = np.full((1, BLOCK), self.cfg.mask_id, dtype=np.int32)
        block_in[0, 0] = self.last
        mask = np.array([(1 << BLOCK) - 1], dtype=np.int64)
        draft = np.full((1, BLOCK), -1, dtype=np.int32)
        for _ in range(steps):
            logits = self.forward(block_in[0], attention.BIDIR)
            ids, conf = self._argmax(logits)
            mask, block_in, draft, _ = decode.unmask(conf[None], ids[None], mask, block_in, draft, k)
        assert int(mask[0]) == 0
        return draft[0]

    def draft_threshold(self, tau: float, tau_revise: float = 2.0) -> np.ndarray:
        block_in = np.full((1, BLOCK), self.cfg.mask_id, dtype=np.int32)
        block_in[0, 0] = self.last
        mask = np.array([(1 << BLOCK) - 1], dtype=np.int64)
        draft = np.full((1, BLOCK), -1, dtype=np.int32)
        tau32, taur32 = float(np.float32(tau)), float(np.float32(tau_revise))
        self.rounds = 0
        while int(mask[0]) != 0:
            logits = self.forward(block_in[0], attention.BIDIR)
            ids, conf = self._argmax(logits)
            conf32 = conf.astype(np.float32).astype(np.float64)
            mask, block_in, draft, _, nr = decode.unmask_threshold(conf32[None], ids[None], mask,
                                                                   block_in, draft, tau32, taur32)
            self.revisions += int(nr[0])
            self.rounds += 1
        return draft[0]

    def _draft_any(self, steps: int, tau):
        return self.draft(steps) if tau is None else self.draft_threshold(*tau)

    def step_diff(self, steps: int, tau=None) -> list[int]:
        d = self._draft_any(steps, tau)
        self.forward([self.last] + [int(t) for t in d[:BLOCK - 1]], attention.BIDIR)
        self.kv_len += BLOCK
        self.last = int(d[BLOCK - 1])
        self.tokens.extend(int(t) for t in d)
        return [int(t) for t in d]

    def step_selfspec(self, steps: int, tau=None) -> list[int]:
        d = self._draft_any(steps, tau)
        logits = self.forward([self.last] + [int(t) for t in d[:BLOCK - 1]], attention.CAUSAL)
        a = self._argmax(logits)[0]
        L, commit, n, _ = decode.verify_accept(d[None], a[None])
        n0 = int(n[0])
        self.accept_lens.append(int(L[0]))
        self.kv_len += n0
        out = [int(t) for t in commit[0, :n0]]
        self.last = out[-1]
        self.tokens.extend(out)
        return out

    def step_selfspec_fused(self) -> list[int]:
        P = self.kv_len
        d = self.pending_draft
        if d is None:
            d = self.draft(1)
        blk = [self.last] + [int(t) for t in d[:BLOCK - 1]]
        a = self._argmax(self.forward(blk, attention.CAUSAL))[0]       # writes KV of [P, P+32)
        # the draft half sees the prefix and the block under verification
        self.kv_len = P + BLOCK
        nxt = self._argmax(self.forward([int(d[BLOCK - 1])] + [self.cfg.mask_id] * (BLOCK - 1),
                                        attention.BIDIR))[0]
        self.kv_len = P
        self.forwards -= 1                      # the two halves are one forward
        L, commit, n, _ = decode.verify_accept(np.asarray(d)[None], a[None])
        n0 = int(n[0])
        self.accept_lens.append(int(L[0]))
        self.kv_len += n0
        out = [int(t) for t in commit[0, :n0]]
        self.last = out[-1]
        self.tokens.extend(out)
        self.pending_draft = nxt if int(L[0]) == BLOCK else None
        return out

    def step_selfspec_quadratic(self, cands) -> list[int]:
        """One cycle of quadratic self-speculation with candidate acceptance
        lengths `cands` (each in [0, 32), besides 32 itself)."""
        P = self.kv_len
        d = self.pending_draft
        if d is None:
            d = self.draft(1)
        blk = [self.last] + [int(t) for t in d[:BLOCK - 1]]
        a = self._argmax(self.forward(blk, attention.CAUSAL))[0]       # writes KV of [P, P+32)
        # the candidate blocks overwrite cache rows past their own prefix;
        # every one of them starts from the verified block's K/V
        saved = [(k[:, P:].copy(), v[:, P:].copy()) for k, v in zip(self.k, self.v)]

        def restore():
            for (k0, v0), k, v in zip(saved, self.k, self.v):
                k[:, P:] = k0
                v[:, P:] = v0

        mask = self.cfg.mask_id
        nxt = {}
        self.kv_len = P + BLOCK
        nxt[BLOCK] = self._argmax(self.forward([int(d[BLOCK - 1])] + [mask] * (BLOCK - 1),
                                               attention.BIDIR))[0]
        for Lc in sorted(set(int(c) for c in cands)):
            assert 0 <= Lc < BLOCK
            restore()
            self.kv_len = P + Lc + 1
            nxt[Lc] = self._argmax(self.forward([mask] * BLOCK, attention.BIDIR))[0]
        restore()
        self.kv_len = P
        self.forwards -= len(nxt)               # verification and all drafts are one forward
        L, commit, n, _ = decode.verify_accept(np.asarray(d)[None], a[None])
        n0, L0 = int(n[0]), int(L[0])
        self.accept_lens.append(L0)
        self.kv_len += n0
        out = [int(t) for t in commit[0, :n0]]
        self.last = out[-1]
        self.tokens.extend(out)
        self.pending_draft = nxt.get(L0)
        return out

    def draft_masked(self) -> np.ndarray:
        """The draft a quadratic candidate block gives from the current state:
        the argmaxes of one BIDIR forward of 32 [MASK] inputs, the pending
        token's slot included."""
        logits = self.forward([self.cfg.mask_id] * BLOCK, attention.BIDIR)
        self.forwards -= 1
        return self._argmax(logits)[0]

    def generate(self, mode: str, n_new: int, steps: int = 1, tau=None, cands=(0, 1)) -> list[int]:
        """Decode until n_new tokens (extra committed tokens are cut). `tau`:
        None for the top-k draft of `steps` rounds, or (tau, tau_revise) for
        the threshold sampler. `cands`: the candidate acceptance lengths of
        quadratic self-speculation."""
        while len(self.tokens) < n_new:
            if mode == "ar":
                self.step_ar()
            elif mode == "diff":
                self.step_diff(steps, tau)
            elif mode == "selfspec":
                self.step_selfspec(steps, tau)
            elif mode == "selfspec-fused":
                self.step_selfspec_fused()
            elif mode == "selfspec-quad":
                self.step_selfspec_quadratic(cands)
            else:
                raise ValueError(mode)
        return self.tokens[:n_new]
