"""Block-causal GQA attention, plain definition, float64.

Follows "Nemotron-Labs-Diffusion: A Tri-Mode Language Model ..." (hotpaper.ai),
technical approach / modules ("Block-wise attention" as the basis of the
diffusion model), and "NVIDIA 发布 Nemotron-Labs Diffusion 语言模型系列"
(fintech-frontier-insights), "三种生成模式" (a 32-token block handled in
parallel) and "训练路线" (block-wise attention keeps the AR model's abilities
and the KV cache). Reading: every block query sees the whole committed prefix;
inside the block it sees every block key (BIDIR, diffusion) or the block keys up
to its own slot (CAUSAL, autoregressive), the split between the two named in
"Nemotron-Labs-Diffusion: 一种统一自回归、扩散和自推测解码的三模式语言模型"
(ai-feeds.com), "问题" (AR needs causal attention, diffusion bidirectional
context).
"""
from __future__ import annotations

import numpy as np

BIDIR = 0
CAUSAL = 1


def visible_count(P: int, T: int, i: int, mode: int) -> int:
    """Number of visible keys (a prefix of cache positions) for block slot i."""
    return P + (i + 1 if mode == CAUSAL else T)


def block_attn(q, k_cache, v_cache, kv_len, mode: int, scale: float, perturb_p=None) -> np.ndarray:
    """q [B][T][Hq][D]; k_cache, v_cache [B][Hkv][Lmax][D]; kv_len [B].

    out[b][i][h] = sum_j p_j v[b][g][j] with p = softmax(scale * q.k_j) over the
    visible keys j of slot i, g = h // (Hq/Hkv). Returns float64 [B][T][Hq][D].
    perturb_p (None for the definition): a function applied to each row's
    probabilities before the product with V, used only by the perturbation
    analysis that derives the bf16 model's tolerance (oracle.model.Perturbation).
    """
    q = np.asarray(q, dtype=np.float64)
    k_cache = np.asarray(k_cache, dtype=np.float64)
    v_cache = np.asarray(v_cache, dtype=np.float64)
    B, T, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    assert Hq % Hkv == 0
    G = Hq // Hkv
    out = np.zeros((B, T, Hq, D), dtype=np.float64)
    for b in range(B):
        P = int(kv_len[b])
        for h in range(Hq):
            g = h // G
            for i in range(T):
                n = visible_count(P, T, i, mode)
                keys = k_cache[b, g, :n]           # [n][D]
                vals = v_cache[b, g, :n]           # [n][D]
                s = scale * (keys @ q[b, i, h])    # [n]
                p = np.exp(s - s.max())
                p /= p.sum()
                if perturb_p is not None:
                    p = perturb_p(p)
                out[b, i, h] = p @ vals
    return out


def block_attn_rows(q, k_cache, v_cache, kv_len, mode: int, scale: float, rows):
    """The same definition evaluated only at the listed (b, i, h) rows; for
    spot checks of full-size launches. Returns float64 [len(rows)][D]."""
    G = q.shape[2] // k_cache.shape[1]
    T = q.shape[1]
    res = []
    for (b, i, h) in rows:
        P = int(kv_len[b])
        g = h // G
        n = visible_count(P, T, i, mode)
        keys = np.asarray(k_cache[b, g, :n], dtype=np.float64)
        vals = np.asarray(v_cache[b, g, :n], dtype=np.float64)
        s = scale * (keys @ np.asarray(q[b, i, h], dtype=np.float64))
        p = np.exp(s - s.max())
        p /= p.sum()
        res.append(p @ vals)
    return np.stack(res)
