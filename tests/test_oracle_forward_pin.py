"""Independent pin of the oracle's model forward (oracle.model.Session.forward).

The same pre-norm transformer is assembled here a second way, from torch
float64 library primitives, and must give the oracle's logits to 1e-12:

- the whole sequence (prefix and block) is recomputed in one pass with an
  explicit attention mask instead of a KV cache filled by a prefill forward;
- RMSNorm is torch.nn.functional.rms_norm, SiLU is torch.nn.functional.silu,
  attention is torch.nn.functional.scaled_dot_product_attention over K/V heads
  replicated to the query heads;
- RoPE is a complex rotation: dims (i, i + D/2) form one complex number that
  is multiplied by exp(1j * pos * base^(-2i/D));
- bf16 rounding (bf16 models) is torch.frexp + round-half-even on 8
  significant bits, not the oracle's bit arithmetic;
- weights are drawn from the Philox stream with the tensor ids and shapes the
  C ABI documents (0 embedding, 1 + 8l + j for layer l with j = 0 q, 1 k, 2 v,
  3 o, 4 gate, 5 up, 6 down, 1 + 8L the LM head), not through oracle.model.

The structure follows the model the pages describe ("NVIDIA 发布 Nemotron-Labs
Diffusion 语言模型系列" (fintech-frontier-insights), "三种生成模式": one
checkpoint for AR, diffusion and self-speculation; "Nemotron-Labs-Diffusion: A
Tri-Mode Language Model ..." (hotpaper.ai), modules: block-wise attention) with
the readings of the design notes (pre-norm, RMSNorm, SwiGLU, rotate-half RoPE,
untied LM head, bf16 rounding points).

A second test plants, one at a time, the mistakes this pin must catch into the
oracle's forward (a dropped residual, gate and up swapped, RoPE on v, the final
norm dropped, k and v tensor ids swapped, ...) and checks that each one fails.
"""
import inspect
import textwrap

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import attention, model, philox
from self_speculative_lm_block_b300 import synth

CONFIGS = {
    "tiny-f32": dict(synth.TINY),
    "gqa-f32": dict(layers=2, d_model=256, n_heads=8, n_kv_heads=2, head_dim=32, ffn=512, vocab=300,
                    dtype="f32", seed=4321),
    "gqa-bf16": dict(layers=2, d_model=256, n_heads=8, n_kv_heads=2, head_dim=64, ffn=384, vocab=300,
                     dtype="bf16", seed=4322),
}


def _ocfg(c):
    return model.Config(layers=c["layers"], d_model=c["d_model"], n_heads=c["n_heads"],
                        n_kv_heads=c["n_kv_heads"], head_dim=c["head_dim"], ffn=c["ffn"],
                        vocab=c["vocab"], dtype=c["dtype"], seed=c["seed"])


def _bf16_round(t: torch.Tensor) -> torch.Tensor:
    """Nearest bf16 value (ties to even) of float64 values: t = m 2^e with
    0.5 <= |m| < 1, and bf16 keeps 8 significant bits, so the grid spacing is
    2^(e-8); torch.round rounds halves to even."""
    m, e = torch.frexp(t)
    return torch.ldexp(torch.round(m * 256.0), e - 8)


def _weight(c, tid, rows, cols):
    w = philox.weight_values(c["seed"], tid, 0, rows * cols).reshape(rows, cols)
    t = torch.from_numpy(w)
    if c["dtype"] == "bf16":
        t = t.to(torch.bfloat16)
    return t.to(torch.float64)


def torch_block_logits(c, prompt, block, causal: bool) -> np.ndarray:
    """Logits [T][V] of the block rows for the sequence prompt[:-1] + block,
    recomputed from scratch; the block starts at position P = len(prompt) - 1."""
    d, Hq, Hkv, D, ffn, V = (c[k] for k in ("d_model", "n_heads", "n_kv_heads", "head_dim", "ffn",
                                            "vocab"))
    L, eps, base = c["layers"], 1e-6, 10000.0
    rb = _bf16_round if c["dtype"] == "bf16" else (lambda t: t)
    ids = [int(t) for t in prompt[:-1]] + [int(t) for t in block]
    P, T = len(prompt) - 1, len(block)
    N = P + T
    # mask[i, j]: query row i may attend to key j
    i = torch.arange(N)[:, None]
    j = torch.arange(N)[None, :]
    in_block = i >= P
    mask = torch.where(in_block, (j < P) | ((j >= P) & ((j <= i) if causal else (j < N))), j <= i)
    pos = torch.arange(N, dtype=torch.float64)
    theta = base ** (-2.0 * torch.arange(D // 2, dtype=torch.float64) / D)
    rot = torch.polar(torch.ones(N, D // 2, dtype=torch.float64), pos[:, None] * theta[None, :])

    def rope(x):  # [N][H][D]
        z = torch.complex(x[..., :D // 2], x[..., D // 2:]) * rot[:, None, :]
        return torch.cat([z.real, z.imag], dim=-1)

    x = _weight(c, 0, V, d)[torch.tensor(ids)]
    for l in range(L):
        t0 = 1 + 8 * l
        h = rb(F.rms_norm(x, (d,), eps=eps))
        q = (h @ _weight(c, t0 + 0, Hq * D, d).T).reshape(N, Hq, D)
        k = (h @ _weight(c, t0 + 1, Hkv * D, d).T).reshape(N, Hkv, D)
        v = (h @ _weight(c, t0 + 2, Hkv * D, d).T).reshape(N, Hkv, D)
        q, k, v = rb(rope(q)), rb(rope(k)), rb(v)
        G = Hq // Hkv
        kq = k.repeat_interleave(G, dim=1)   # query head hh reads kv head hh // G
        vq = v.repeat_interleave(G, dim=1)
        o = F.scaled_dot_product_attention(q.transpose(0, 1), kq.transpose(0, 1), vq.transpose(0, 1),
                                           attn_mask=mask, scale=1.0 / np.sqrt(D))
        o = rb(o.transpose(0, 1).reshape(N, Hq * D))
        x = x + o @ _weight(c, t0 + 3, d, Hq * D).T
        h = rb(F.rms_norm(x, (d,), eps=eps))
        g = h @ _weight(c, t0 + 4, ffn, d).T
        u = h @ _weight(c, t0 + 5, ffn, d).T
        a = rb(F.silu(g) * u)
        x = x + a @ _weight(c, t0 + 6, d, ffn).T
    h = rb(F.rms_norm(x, (d,), eps=eps))
    logits = h @ _weight(c, 1 + 8 * L, V, d).T
    return logits[P:].numpy()


def _inputs(c, T, seed):
    V = c["vocab"]
    prompt = [int(t) for t in synth.prompt(9, V, seed)]
    block = [prompt[-1]] + [int(t) for t in synth.prompt(T - 1, V, seed + 1)]
    return prompt, block


def _oracle_block_logits(c, prompt, block, mode, weights=None):
    cfg = _ocfg(c)
    s = model.Session(cfg, weights or model.Weights(cfg), max_seq=64)
    s.prefill(prompt)
    return s.forward(block, mode)


def _rel_err(a, b):
    return float(np.abs(a - b).max() / max(1.0, np.abs(b).max()))


@pytest.mark.parametrize("name", list(CONFIGS))
@pytest.mark.parametrize("T", [1, 12, 32])
def test_oracle_forward_equals_independent_assembly(name, T):
    c = CONFIGS[name]
    prompt, block = _inputs(c, T, 31 + T)
    w = model.Weights(_ocfg(c))
    for mode in (attention.BIDIR, attention.CAUSAL):
        ref = torch_block_logits(c, prompt, block, causal=(mode == attention.CAUSAL))
        got = _oracle_block_logits(c, prompt, block, mode, w)
        assert got.shape == ref.shape
        assert _rel_err(got, ref) <= 1e-12, (name, T, mode, _rel_err(got, ref))


def test_bf16_rounding_of_the_pin_is_nearest_even():
    """The pin's own rounding: grid points stay, midpoints go to the even
    neighbour, other values to the nearer neighbour, carries move the exponent."""
    x = torch.tensor([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -8 + 2 ** -30,
                      -(2.0 - 2 ** -9), 3.0 * 2 ** -130, 0.0], dtype=torch.float64)
    want = [1.0, 1.0, 1.0 + 4 * 2 ** -8, 1.0 + 2 ** -7, -2.0, 3.0 * 2 ** -130, 0.0]
    assert _bf16_round(x).tolist() == want
    y = torch.randn(10000, dtype=torch.float64, generator=torch.Generator().manual_seed(0)) * 5
    r = _bf16_round(y)
    # on the bf16 grid, and within half a spacing of the input
    assert torch.equal(r.float().to(torch.bfloat16).double(), r)
    _, e = torch.frexp(y)
    assert (torch.abs(r - y) <= torch.ldexp(torch.ones_like(y), e - 9)).all()


# ---------------------------------------------------------------- planted mistakes
_KV_SWAP = ("w.full(tid_layer(l, 1))", "w.full(tid_layer(l, 2))")
MUTATIONS = {
    "attention residual dropped": [("x = x + rowwise_matmul(o,", "x = rowwise_matmul(o,")],
    "ffn residual dropped": [("x = x + rowwise_matmul(a,", "x = rowwise_matmul(a,")],
    "gate and up swapped": [("silu(g) * u", "silu(u) * g")],
    "rope applied to v": [("v = self._rb(v)", "v = self._rb(rope(v, pos, cfg.rope_base))")],
    "rope dropped on k": [("k = self._rb(rope(k, pos, cfg.rope_base))", "k = self._rb(k)")],
    "final norm dropped": [("h = self._rb(rmsnorm(x, cfg.eps))\n    wl", "h = self._rb(x)\n    wl")],
    "k and v tensor ids swapped": [(_KV_SWAP[0], "@@K@@"), (_KV_SWAP[1], _KV_SWAP[0]),
                                   ("@@K@@", _KV_SWAP[1])],
    "mask mode inverted": [("[P], mode,", "[P], 1 - mode,")],
    "attention scale dropped": [("1.0 / np.sqrt(D))[0]", "1.0)[0]")],
}


def _mutated_forward(edits):
    src = textwrap.dedent(inspect.getsource(model.Session.forward))
    for old, new in edits:
        assert src.count(old) == 1, f"mutation anchor not found once: {old!r}"
        src = src.replace(old, new)
    ns = dict(vars(model))
    exec(compile(src, "<mutated oracle forward>", "exec"), ns)
    return ns["forward"]


@pytest.mark.parametrize("mutation", list(MUTATIONS))
def test_pin_catches_planted_mistakes(mutation, monkeypatch):
    c = CONFIGS["gqa-bf16"]
    prompt, block = _inputs(c, 12, 77)
    w = model.Weights(_ocfg(c))
    refs = {m: torch_block_logits(c, prompt, block, causal=(m == attention.CAUSAL))
            for m in (attention.BIDIR, attention.CAUSAL)}
    # unmutated: both modes agree with the pin
    for m, ref in refs.items():
        assert _rel_err(_oracle_block_logits(c, prompt, block, m, w), ref) <= 1e-12
    monkeypatch.setattr(model.Session, "forward", _mutated_forward(MUTATIONS[mutation]))
    worst = max(_rel_err(_oracle_block_logits(c, prompt, block, m, w), ref) for m, ref in refs.items())
    assert worst > 1e-6, (mutation, worst)
