"""Logits reduction, diffusion unmask step and self-speculation verify/accept.

Plain definitions in Python/NumPy, float64 where floating point is involved.

- Greedy decision: temperature 0 is the setting under which self-speculation
  reproduces AR output ("NVIDIA 发布 Nemotron-Labs Diffusion 语言模型系列"
  (fintech-frontier-insights), "三种生成模式" and "准确性"), so every mode picks
  the argmax. Reading: ties go to the lowest id; the [MASK] id is excluded.
- Confidence: the probability of the chosen id under the full softmax (the
  excluded id is part of the normaliser).
- Unmask: one denoising round of the 32-token block ("三种生成模式": several
  rounds of iterative denoising per block). Reading: among still-masked slots,
  the k highest-confidence ones are fixed (ties to the lower slot), without
  remasking.
- Threshold unmask with revision (sampler variants): "NVIDIA 发布
  Nemotron-Labs Diffusion：三模态语言模型统一 AR 与扩散解码" (aimodeling.com
  digest of the Hugging Face blog): the refinement steps are a budget the user
  can lower, and the diffusion model can revise tokens it already produced;
  "Nemotron-Labs-Diffusion: 一种统一自回归、扩散和自推测解码的三模式语言模型"
  (ai-feeds.com), 核心洞察: the sampler decides the tokens per forward.
  Reading: a round fixes every masked slot whose confidence reaches tau (at
  least the single most confident one, ties to the lower slot, so each round
  makes progress), and, before that, replaces the token of every slot fixed in
  an earlier round whose current prediction differs with confidence at least
  tau_revise (tau_revise > 1 turns revision off).
- Verify/accept: gsyq.cn explainer, §2.3 "自推测解码": the verifier accepts the
  agreeing prefix, rejects the first mismatching draft and everything after it,
  and supplies its own token at that position.
"""
from __future__ import annotations

import numpy as np


def logits_reduce(logits, V: int | None = None, exclude_id: int = -1):
    """logits [R][>=V] -> (argmax int32 [R], conf float64 [R])."""
    x = np.asarray(logits, dtype=np.float64)
    R = x.shape[0]
    V = x.shape[1] if V is None else V
    ids = np.empty(R, dtype=np.int32)
    conf = np.empty(R, dtype=np.float64)
    for r in range(R):
        row = x[r, :V]
        cand = row.copy()
        if 0 <= exclude_id < V:
            cand[exclude_id] = -np.inf
        if V == 0 or np.all(np.isneginf(cand)):
            ids[r], conf[r] = -1, 0.0
            continue
        best = int(np.argmax(cand))           # first occurrence = lowest id
        m = row.max()
        z = np.exp(row - m).sum()
        ids[r] = best
        conf[r] = np.exp(row[best] - m) / z
    return ids, conf


def unmask(conf, pred, mask_bits, block_in, draft, k: int):
    """One unmask round over [B][T] slots. Returns updated copies
    (mask_bits, block_in, draft) and chosen [B][k] (-1 padded)."""
    conf = np.asarray(conf)
    pred = np.asarray(pred)
    B, T = conf.shape
    mask_bits = np.array(mask_bits, dtype=np.int64) & ((1 << T) - 1 if T < 64 else -1)
    block_in = np.array(block_in, dtype=np.int32)
    draft = np.array(draft, dtype=np.int32)
    chosen = np.full((B, k), -1, dtype=np.int32)
    for b in range(B):
        masked = [i for i in range(T) if (int(mask_bits[b]) >> i) & 1]
        order = sorted(masked, key=lambda i: (-float(conf[b, i]), i))
        for r, i in enumerate(order[:k]):
            chosen[b, r] = i
            draft[b, i] = pred[b, i]
            mask_bits[b] &= ~(1 << i)
            if i <= T - 2:
                block_in[b, i + 1] = pred[b, i]
    return mask_bits.astype(np.uint32), block_in, draft, chosen


def unmask_threshold(conf, pred, mask_bits, block_in, draft, tau: float, tau_revise: float = 2.0):
    """One threshold round over [B][T] slots. Returns updated copies
    (mask_bits, block_in, draft) and per sequence the number of slots fixed
    and the number of earlier slots revised."""
    conf = np.asarray(conf, dtype=np.float64)
    pred = np.asarray(pred)
    B, T = conf.shape
    mask_bits = np.array(mask_bits, dtype=np.int64) & ((1 << T) - 1)
    block_in = np.array(block_in, dtype=np.int32)
    draft = np.array(draft, dtype=np.int32)
    n_fixed = np.zeros(B, dtype=np.int32)
    n_revised = np.zeros(B, dtype=np.int32)
    for b in range(B):
        mask = int(mask_bits[b])
        masked = [i for i in range(T) if (mask >> i) & 1]
        earlier = [i for i in range(T) if not (mask >> i) & 1]
        # revision of slots fixed in earlier rounds
        for i in earlier:
            if pred[b, i] != draft[b, i] and conf[b, i] >= tau_revise:
                draft[b, i] = pred[b, i]
                if i <= T - 2:
                    block_in[b, i + 1] = pred[b, i]
                n_revised[b] += 1
        # every masked slot at or above tau; else the most confident one
        chosen = [i for i in masked if conf[b, i] >= tau]
        if not chosen and masked:
            best = masked[0]
            for i in masked[1:]:
                if conf[b, i] > conf[b, best]:
                    best = i
            chosen = [best]
        for i in chosen:
            draft[b, i] = pred[b, i]
            mask &= ~(1 << i)
            if i <= T - 2:
                block_in[b, i + 1] = pred[b, i]
        mask_bits[b] = mask
        n_fixed[b] = len(chosen)
    return mask_bits.astype(np.uint32), block_in, draft, n_fixed, n_revised


def verify_accept(draft, target, kv_len=None):
    """Returns (accept_len [B], commit [B][T] (-1 padded), n_commit [B],
    kv_len' [B] or None)."""
    draft = np.asarray(draft)
    target = np.asarray(target)
    B, T = draft.shape
    L = np.empty(B, dtype=np.int32)
    n = np.empty(B, dtype=np.int32)
    commit = np.full((B, T), -1, dtype=np.int32)
    for b in range(B):
        i = 0
        while i < T and draft[b, i] == target[b, i]:
            i += 1
        L[b] = i
        n[b] = min(i + 1, T)
        commit[b, : n[b]] = target[b, : n[b]]
    new_len = None if kv_len is None else np.asarray(kv_len, dtype=np.int32) + n
    return L, commit, n, new_len
