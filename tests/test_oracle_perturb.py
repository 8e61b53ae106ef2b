"""The perturbation analysis that sets the bf16 model's logit tolerance
(oracle.perturb): with zero noise its forward is the oracle's forward, with the
GPU's error model it moves the logits by a nonzero, finite amount, and the bar
it derives scales with each logit's LM-head row."""
import numpy as np
import pytest

from oracle import attention, model, perturb
from self_speculative_lm_block_b300 import synth

CFGS = {
    "bf16": dict(layers=2, d_model=256, n_heads=4, n_kv_heads=2, head_dim=64, ffn=512, vocab=700,
                 dtype="bf16", seed=5),
    "f32": dict(synth.TINY),
}


def _cfg(c):
    return model.Config(layers=c["layers"], d_model=c["d_model"], n_heads=c["n_heads"],
                        n_kv_heads=c["n_kv_heads"], head_dim=c["head_dim"], ffn=c["ffn"],
                        vocab=c["vocab"], dtype=c["dtype"], seed=c["seed"])


@pytest.mark.parametrize("name", list(CFGS))
def test_zero_noise_forward_is_the_oracle(name):
    cfg = _cfg(CFGS[name])
    w = model.Weights(cfg)
    pr = synth.prompt(20, cfg.vocab, 3)
    blk = [int(pr[-1])] + [int(t) for t in synth.prompt(31, cfg.vocab, 4)]
    for mode in (attention.BIDIR, attention.CAUSAL):
        a = model.Session(cfg, w, max_seq=64)
        a.prefill(pr)
        b = perturb.PerturbedSession(cfg, w, 64, perturb.Perturbation(0, 0.0, 0.0, 0.0, 0.0))
        b.prefill(pr)
        ra, rb = a.forward(blk, mode), b.forward(blk, mode)
        assert np.abs(ra - rb).max() <= 1e-12 * np.abs(ra).max()


def test_noise_moves_the_logits_and_the_bar_follows_the_rows():
    cfg = _cfg(CFGS["bf16"])
    w = model.Weights(cfg)
    pr = synth.prompt(20, cfg.vocab, 3)
    blk = [int(pr[-1])] + [int(t) for t in synth.prompt(31, cfg.vocab, 4)]
    ref, bar = perturb.logit_bar(cfg, w, pr, blk, attention.CAUSAL, runs=3, max_seq=64)
    s = model.Session(cfg, w, max_seq=64)
    s.prefill(pr)
    assert np.array_equal(s.forward(blk, attention.CAUSAL), ref)
    assert np.isfinite(bar).all() and (bar > 0).all()
    # well below the logits' own size, and far above fp32 rounding of them
    mr = np.abs(ref).max(axis=-1, keepdims=True)
    assert (bar < 0.1 * mr).all() and (bar > 1e-5 * mr).all()
    # one perturbed rerun stays inside the bar (it is one draw of the same noise)
    p = perturb.PerturbedSession(cfg, w, 64, perturb.Perturbation(99))
    p.prefill(pr)
    assert (np.abs(p.forward(blk, attention.CAUSAL) - ref) <= bar).all()
    # the scale of row t, logit n is ||W_lm[n] * h_t||: doubling one LM-head
    # row doubles that logit's bar
    wl = w.full(model.tid_lm(cfg)).copy()
    w._cache[model.tid_lm(cfg)][7] *= 2.0
    try:
        _, bar2 = perturb.logit_bar(cfg, w, pr, blk, attention.CAUSAL, runs=3, max_seq=64)
    finally:
        w._cache[model.tid_lm(cfg)][:] = wl
    ratio = bar2[:, 7] / bar[:, 7]
    assert np.all((ratio > 1.5) & (ratio < 2.5))


def test_teacher_forced_ar_bars_follow_given_tokens():
    cfg = _cfg(CFGS["bf16"])
    w = model.Weights(cfg)
    pr = synth.prompt(16, cfg.vocab, 8)
    s = model.Session(cfg, w, max_seq=64)
    s.prefill(pr)
    toks = s.generate("ar", 6)
    steps = perturb.ar_reference_with_bars(cfg, w, pr, toks, runs=2)
    assert len(steps) == 6
    for (ref, bar), t in zip(steps, toks):
        row = ref.copy()
        row[cfg.mask_id] = -np.inf
        assert int(np.argmax(row)) == t     # the oracle's own tokens are its argmaxes
        assert (bar > 0).all()
