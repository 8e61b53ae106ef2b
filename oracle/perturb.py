"""Perturbation analysis of the bf16 model: the scale of the tolerance for
comparisons of a GPU forward with the oracle's.

Test infrastructure (tests only). The oracle computes the bf16 model in
float64 and rounds to bf16 at the points the design fixes (weights, the inputs
of every matrix product, q/k/v). A GPU computes the same model in fp32 with
another order of accumulation, with bf16 attention probabilities and with fast
fp32 functions. So the values it rounds to bf16 differ from the oracle's in
their last fp32 bits, some roundings land on the neighbouring bf16 value, and
those differences travel through the layers to the logits. How far the logits
move under differences of that size is measured here by Monte Carlo arithmetic
(D. Stott Parker, "Monte Carlo Arithmetic: exploiting randomness in
floating-point arithmetic", UCLA CSD-970002, 1997). The forward is rerun
several times, each time with fresh random noise of the GPU's error size at
every place where the GPU computes differently, and the spread of the logits
over the runs sets the scale of the tolerance (`logit_bar`).

Error model of the GPU (the size of each injected term):
- a matrix product y_n = sum_k x_k w_nk accumulated in fp32: Gaussian
  absolute noise with standard deviation u sqrt(K) ||x * w_n||_2, u = 2^-24.
  This is about ten times the standard deviation of a sequential fp32 sum of
  such terms (u sqrt(K / 96) ||x * w_n||_2 for K/16 accumulations of 16 products).
  The GPU tests of the projection kernel check its error against 8 of these
  standard deviations, element by element;
- attention probabilities rounded to bf16 before the product with V: each
  probability times (1 + e), e uniform in [-2^-9, 2^-9], the bound of one
  round-to-nearest-even onto 8 significant bits;
- fp32 RMSNorm, RoPE, SiLU and attention output: relative noise uniform in
  [-2^-22, 2^-22] (a few fp32 ulps);
- the fp32 residual stream: relative noise uniform in [-2^-24, 2^-24] after
  each addition (one fp32 rounding).
With every amplitude set to zero the perturbed forward is the oracle's forward
(a CPU test checks this to 1e-12).
"""
from __future__ import annotations

import numpy as np

from . import attention
from .model import Session, rmsnorm, rope, silu, tid_embed, tid_layer, tid_lm

U32 = 2.0 ** -24


class Perturbation:
    """One run's noise source and amplitudes (see the module docstring)."""

    def __init__(self, seed: int, gemm: float = 1.0, prob: float = 2.0 ** -9, fn: float = 2.0 ** -22,
                 resid: float = U32):
        self.rng = np.random.default_rng(seed)
        self.gemm, self.prob, self.fn, self.resid = gemm, prob, fn, resid

    def rel(self, x, eps: float):
        if eps == 0.0:
            return x
        return x * (1.0 + self.rng.uniform(-eps, eps, size=np.shape(x)))

    def matmul(self, x: np.ndarray, w: np.ndarray) -> np.ndarray:
        """x [T][K] times w [N][K]^T, plus the accumulation noise of each output."""
        y = x @ w.T
        if self.gemm == 0.0:
            return y
        K = x.shape[-1]
        s = np.sqrt((x * x) @ (w * w).T)
        return y + self.rng.standard_normal(y.shape) * (self.gemm * U32 * np.sqrt(K)) * s


class PerturbedSession(Session):
    """The oracle's session with the forward rerun under a Perturbation. The
    layer is assembled exactly as in oracle.model.Session.forward; only the
    noise terms are added. `last_hidden` keeps the final normed hidden state."""

    def __init__(self, cfg, weights=None, max_seq: int = 4096, perturb: Perturbation | None = None):
        super().__init__(cfg, weights, max_seq)
        self.pz = perturb or Perturbation(0, 0.0, 0.0, 0.0, 0.0)
        self.last_hidden = None

    def forward(self, ids, mode: int, vocab_rows=None) -> np.ndarray:
        cfg, w, pz = self.cfg, self.w, self.pz
        ids = np.asarray(ids, dtype=np.int64)
        T = ids.shape[0]
        P = self.kv_len
        D, Hq, Hkv = cfg.head_dim, cfg.n_heads, cfg.n_kv_heads
        pos = np.arange(P, P + T)
        x = w.rows(tid_embed(), ids)
        for l in range(cfg.layers):
            h = self._rb(pz.rel(rmsnorm(x, cfg.eps), pz.fn))
            q = pz.matmul(h, w.full(tid_layer(l, 0))).reshape(T, Hq, D)
            k = pz.matmul(h, w.full(tid_layer(l, 1))).reshape(T, Hkv, D)
            v = pz.matmul(h, w.full(tid_layer(l, 2))).reshape(T, Hkv, D)
            q = self._rb(rope(pz.rel(q, pz.fn), pos, cfg.rope_base))
            k = self._rb(rope(pz.rel(k, pz.fn), pos, cfg.rope_base))
            v = self._rb(v)
            self.k[l][:, P:P + T] = k.transpose(1, 0, 2)
            self.v[l][:, P:P + T] = v.transpose(1, 0, 2)
            o = attention.block_attn(q[None], self.k[l][None], self.v[l][None], [P], mode,
                                     1.0 / np.sqrt(D), lambda p: pz.rel(p, pz.prob))[0]
            o = self._rb(pz.rel(o, pz.fn)).reshape(T, Hq * D)
            x = pz.rel(x + pz.matmul(o, w.full(tid_layer(l, 3))), pz.resid)
            h = self._rb(pz.rel(rmsnorm(x, cfg.eps), pz.fn))
            g = pz.matmul(h, w.full(tid_layer(l, 4)))
            u = pz.matmul(h, w.full(tid_layer(l, 5)))
            a = self._rb(pz.rel(silu(g) * u, pz.fn))
            x = pz.rel(x + pz.matmul(a, w.full(tid_layer(l, 6))), pz.resid)
        h = self._rb(pz.rel(rmsnorm(x, cfg.eps), pz.fn))
        self.last_hidden = h
        wl = w.full(tid_lm(cfg)) if vocab_rows is None else w.rows(tid_lm(cfg), vocab_rows)
        self.forwards += 1
        return pz.matmul(h, wl)


def _lm_rows(cfg, weights, vocab_rows):
    return weights.full(tid_lm(cfg)) if vocab_rows is None else weights.rows(tid_lm(cfg), vocab_rows)


def logit_bar(cfg, weights, prompt, block, mode: int, vocab_rows=None, runs: int = 6, z: float = 6.0,
              seed: int = 0, max_seq: int = 512):
    """Reference logits of `block` after prefilling `prompt` (the unperturbed
    forward, equal to the oracle's) and an element-wise bar for a GPU's logits:

        bar[t][n] = z * rho_t * s_tn,   s_tn = || W_lm[n] * h_t ||_2,

    h_t the final normed hidden state of row t, and rho_t the largest over the
    runs of the root mean square over n of (logits_run - ref)[t][n] / s_tn. The
    deviation of logit n is a sum over k of W_lm[n][k] times the hidden-state
    deviation k, so its scale follows || W_lm[n] * h_t ||; rho_t measures how
    large the hidden-state deviations are relative to h_t. z = 6 leaves a
    Gaussian tail of 2e-9 per element."""
    ref_s = PerturbedSession(cfg, weights, max_seq)
    ref_s.prefill(prompt)
    ref = ref_s.forward(block, mode, vocab_rows)
    h = ref_s.last_hidden
    wl = _lm_rows(cfg, weights, vocab_rows)
    s = np.sqrt((h * h) @ (wl * wl).T)
    s = np.where(s > 0, s, 1.0)
    rho = np.zeros(ref.shape[0])
    for r in range(runs):
        ps = PerturbedSession(cfg, weights, max_seq, Perturbation(seed * 1000 + r + 1))
        ps.prefill(prompt)
        d = (ps.forward(block, mode, vocab_rows) - ref) / s
        rho = np.maximum(rho, np.sqrt(np.mean(d * d, axis=-1)))
    return ref, z * rho[:, None] * s


def ar_reference_with_bars(cfg, weights, prompt, tokens, runs: int = 6, z: float = 6.0, seed: int = 0):
    """Teacher-forced AR reference for a given token sequence (a GPU's output):
    for each step i the oracle's logits [V] after prompt + tokens[:i] and the
    element-wise bar of `logit_bar`, all sessions fed the same given tokens."""
    n = len(tokens)
    max_seq = len(prompt) + n + 8
    sessions = [PerturbedSession(cfg, weights, max_seq)] + [
        PerturbedSession(cfg, weights, max_seq, Perturbation(seed * 1000 + r + 1)) for r in range(runs)]
    for s in sessions:
        s.prefill(prompt)
    wl = weights.full(tid_lm(cfg))
    out = []
    for i in range(n):
        logits = []
        for s in sessions:
            logits.append(s.forward([s.last], attention.CAUSAL)[0])
            s.kv_len += 1
            s.last = int(tokens[i])
        h = sessions[0].last_hidden[0]
        sc = np.sqrt((wl * wl) @ (h * h))
        sc = np.where(sc > 0, sc, 1.0)
        rho = max(float(np.sqrt(np.mean(((lg - logits[0]) / sc) ** 2))) for lg in logits[1:]) if runs else 0.0
        out.append((logits[0], z * rho * sc))
    return out
