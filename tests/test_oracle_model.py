"""Pins of the oracle model: component closed forms (RMSNorm, RoPE, SiLU), the
row independence that makes temperature-0 self-speculation equal AR, exact
self-spec == AR on the tiny configuration, forced acceptance, and the stored
tiny-configuration tokens (written by tests/golden/make_golden.py from the
oracle alone)."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import attention, model
from self_speculative_lm_block_b300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tiny_tokens.json")


def tiny_cfg():
    t = synth.TINY
    return model.Config(layers=t["layers"], d_model=t["d_model"], n_heads=t["n_heads"],
                        n_kv_heads=t["n_kv_heads"], head_dim=t["head_dim"], ffn=t["ffn"],
                        vocab=t["vocab"], dtype="f32", seed=t["seed"])


def test_rmsnorm_closed_form_and_library():
    x = np.full((1, 16), -3.0)
    np.testing.assert_allclose(model.rmsnorm(x, 1e-6), -3 / np.sqrt(9 + 1e-6), rtol=1e-15)
    y = np.random.default_rng(0).standard_normal((4, 64))
    ref = torch.nn.functional.rms_norm(torch.from_numpy(y), (64,), eps=1e-6).numpy()
    np.testing.assert_allclose(model.rmsnorm(y, 1e-6), ref, rtol=1e-13)


def test_rope_properties():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((1, 3, 32))
    k = rng.standard_normal((1, 3, 32))
    # position 0 is the identity; rotations keep norms
    assert np.allclose(model.rope(q, [0], 10000.0), q, rtol=0, atol=0)
    r = model.rope(q, [77], 10000.0)
    np.testing.assert_allclose(np.linalg.norm(r, axis=-1), np.linalg.norm(q, axis=-1), rtol=1e-13)
    # scores depend only on the relative position m - n
    def score(m, n):
        return np.sum(model.rope(q, [m], 10000.0) * model.rope(k, [n], 10000.0), axis=-1)
    np.testing.assert_allclose(score(10, 3), score(107, 100), rtol=1e-10)
    # rotate-half pairing: a vector with only component i rotates into i + D/2
    e = np.zeros((1, 1, 32)); e[0, 0, 2] = 1.0
    th = 5 * 10000.0 ** (-4 / 32)
    out = model.rope(e, [5], 10000.0)[0, 0]
    assert abs(out[2] - np.cos(th)) < 1e-15 and abs(out[18] - np.sin(th)) < 1e-15
    assert np.count_nonzero(np.abs(out) > 1e-15) == 2


def test_silu_library():
    x = np.linspace(-8, 8, 101)
    np.testing.assert_allclose(model.silu(x), torch.nn.functional.silu(torch.from_numpy(x)).numpy(),
                               rtol=1e-14, atol=1e-16)


def test_forward_rows_do_not_depend_on_block_length():
    cfg = tiny_cfg()
    w = model.Weights(cfg)
    ids = synth.prompt(20, cfg.vocab, 5)
    s = model.Session(cfg, w, max_seq=64)
    s.prefill(ids[:9])                    # cache holds ids[0..7], last = ids[8]
    blk = s.forward(list(ids[8:20]), attention.CAUSAL)
    for i in range(12):
        s1 = model.Session(cfg, w, max_seq=64)
        s1.prefill(ids[:9 + i])           # cache holds ids[0..7+i], last = ids[8+i]
        one = s1.forward([int(ids[8 + i])], attention.CAUSAL)
        assert np.array_equal(one[0], blk[i])


@pytest.mark.parametrize("steps", [1, 2, 4])
def test_selfspec_equals_ar_exactly(steps):
    cfg = tiny_cfg()
    w = model.Weights(cfg)
    pr = synth.prompt(32, cfg.vocab, cfg.seed)
    s = model.Session(cfg, w, max_seq=200); s.prefill(pr)
    ar = s.generate("ar", 64)
    s2 = model.Session(cfg, w, max_seq=200); s2.prefill(pr)
    assert s2.generate("selfspec", 64, steps) == ar


def test_forced_accept_gives_full_block():
    """Drafting the AR continuation itself is accepted whole (L = 32)."""
    cfg = tiny_cfg()
    w = model.Weights(cfg)
    pr = synth.prompt(32, cfg.vocab, cfg.seed)
    s = model.Session(cfg, w, max_seq=200); s.prefill(pr)
    ar = s.generate("ar", 40)
    s2 = model.Session(cfg, w, max_seq=200); s2.prefill(pr)
    logits = s2.forward([s2.last] + ar[:31], attention.CAUSAL)
    a = model.decode.logits_reduce(logits, exclude_id=cfg.mask_id)[0]
    assert list(a) == ar[:32]


def test_diff_mode_fills_every_slot_and_counts_forwards():
    cfg = tiny_cfg()
    pr = synth.prompt(32, cfg.vocab, cfg.seed)
    for steps in (1, 4, 32):
        s = model.Session(cfg, max_seq=200); s.prefill(pr)
        toks = s.generate("diff", 64, steps)
        assert len(toks) == 64 and all(0 <= t < cfg.vocab - 1 for t in toks)
        assert s.forwards == 2 * (steps + 1)
        assert s.kv_len == 31 + 64


def test_golden_tiny_tokens():
    with open(GOLDEN) as f:
        g = json.load(f)
    cfg = tiny_cfg()
    w = model.Weights(cfg)
    pr = synth.prompt(32, cfg.vocab, cfg.seed)
    assert g["prompt"] == [int(t) for t in pr]
    for key, (mode, steps) in {"ar": ("ar", 1), "diff_k4": ("diff", 8), "selfspec_s1": ("selfspec", 1)}.items():
        s = model.Session(cfg, w, max_seq=200); s.prefill(pr)
        assert s.generate(mode, 64, steps) == g[key], key


# ---------------------------------------------------------------- threshold sampler
def test_threshold_sampler_special_cases_reduce_to_topk():
    """tau above 1 fixes one slot per round: the top-k draft with 32 rounds;
    tau 0 fixes every slot in the first round: the top-k draft with 1 round."""
    cfg = tiny_cfg()
    w = model.Weights(cfg)
    pr = synth.prompt(32, cfg.vocab, cfg.seed)
    for steps, tau in ((32, (1.5, 2.0)), (1, (0.0, 2.0))):
        a = model.Session(cfg, w, max_seq=200); a.prefill(pr)
        b = model.Session(cfg, w, max_seq=200); b.prefill(pr)
        assert a.generate("diff", 64, steps) == b.generate("diff", 64, tau=tau)
        assert a.forwards == b.forwards == 2 * (steps + 1)


@pytest.mark.parametrize("tau", [(0.05, 2.0), (0.02, 0.5), (0.3, 0.0)])
def test_threshold_selfspec_equals_ar(tau):
    """Whatever the draft sampler, verification makes self-speculation emit
    the AR tokens."""
    cfg = tiny_cfg()
    w = model.Weights(cfg)
    pr = synth.prompt(32, cfg.vocab, cfg.seed)
    s = model.Session(cfg, w, max_seq=200); s.prefill(pr)
    ar = s.generate("ar", 48)
    s2 = model.Session(cfg, w, max_seq=200); s2.prefill(pr)
    assert s2.generate("selfspec", 48, tau=tau) == ar


def test_threshold_diff_rounds_and_revisions():
    """A mid threshold takes between 1 and 32 rounds per block; tau_revise 0
    revises every earlier slot whose prediction changed, so revisions happen;
    every committed id is a real token."""
    cfg = tiny_cfg()
    pr = synth.prompt(32, cfg.vocab, cfg.seed)
    s = model.Session(cfg, max_seq=200); s.prefill(pr)
    toks = s.generate("diff", 64, tau=(0.05, 0.0))
    assert len(toks) == 64 and all(0 <= t < cfg.vocab - 1 for t in toks)
    assert 2 * 2 <= s.forwards <= 2 * 33
    assert s.revisions > 0


# ---------------------------------------------------------------- fused self-speculation
def _cfg_vocab(V, seed=7):
    t = synth.TINY
    return model.Config(layers=t["layers"], d_model=t["d_model"], n_heads=t["n_heads"],
                        n_kv_heads=t["n_kv_heads"], head_dim=t["head_dim"], ffn=t["ffn"],
                        vocab=V, dtype="f32", seed=seed)


def test_fused_selfspec_equals_ar():
    cfg = tiny_cfg()
    w = model.Weights(cfg)
    pr = synth.prompt(32, cfg.vocab, cfg.seed)
    s = model.Session(cfg, w, max_seq=260); s.prefill(pr)
    ar = s.generate("ar", 64)
    s2 = model.Session(cfg, w, max_seq=260); s2.prefill(pr)
    assert s2.generate("selfspec-fused", 64) == ar


def test_fused_full_acceptance_takes_one_forward_per_block():
    """With two ids ([MASK] and one token) every draft is accepted: one drafting
    forward, then one fused forward per 32 tokens."""
    cfg = _cfg_vocab(2)
    w = model.Weights(cfg)
    s = model.Session(cfg, w, max_seq=260); s.prefill([0] * 20)
    toks = s.generate("selfspec-fused", 96)
    assert toks == [0] * 96
    assert s.forwards == 1 + 3 and s.accept_lens == [32, 32, 32]
    assert s.kv_len == 19 + 96


def test_fused_next_draft_is_the_draft_of_the_new_state():
    """After a fully accepted block, the draft the fused forward leaves is the
    one a fresh drafting forward computes from the committed tokens (same
    positions and prefix: the shifted block layout holds across the two halves);
    with eight ids full acceptances happen and mix with partial ones, and the
    tokens stay the AR tokens."""
    cfg = _cfg_vocab(8, seed=11)
    w = model.Weights(cfg)
    pr = [int(x) for x in synth.prompt(24, cfg.vocab, 5)]
    s = model.Session(cfg, w, max_seq=600); s.prefill(pr)
    ar = s.generate("ar", 160)
    f = model.Session(cfg, w, max_seq=600); f.prefill(pr)
    checked = 0
    while len(f.tokens) < 160:
        f.step_selfspec_fused()
        if f.pending_draft is not None and checked < 3:
            fresh = model.Session(cfg, w, max_seq=600)
            fresh.prefill(pr + f.tokens)
            assert np.array_equal(fresh.draft(1), f.pending_draft)
            checked += 1
    assert f.tokens[:160] == ar
    assert 32 in f.accept_lens and min(f.accept_lens) < 32
    assert checked >= 1


# ---------------------------------------------------------------- quadratic self-speculation
@pytest.mark.parametrize("cands", [(0, 1), (0, 5, 31), ()])
def test_quadratic_selfspec_equals_ar(cands):
    cfg = tiny_cfg()
    w = model.Weights(cfg)
    pr = synth.prompt(32, cfg.vocab, cfg.seed)
    s = model.Session(cfg, w, max_seq=400); s.prefill(pr)
    ar = s.generate("ar", 64)
    q = model.Session(cfg, w, max_seq=400); q.prefill(pr)
    assert q.generate("selfspec-quad", 64, cands=cands) == ar


def test_quadratic_with_every_candidate_drafts_once():
    """Candidates 0..31 plus full acceptance cover every outcome, so only the
    first cycle runs a drafting forward: forwards = cycles + 1."""
    cfg = _cfg_vocab(8, seed=11)
    w = model.Weights(cfg)
    pr = [int(x) for x in synth.prompt(24, cfg.vocab, 5)]
    s = model.Session(cfg, w, max_seq=900); s.prefill(pr)
    ar = s.generate("ar", 96)
    q = model.Session(cfg, w, max_seq=900); q.prefill(pr)
    assert q.generate("selfspec-quad", 96, cands=tuple(range(32))) == ar
    assert q.forwards == len(q.accept_lens) + 1
    assert min(q.accept_lens) < 32


def test_quadratic_full_acceptance_is_linear():
    """Two ids: every draft is accepted; the quadratic mode then behaves as the
    linear one (one drafting forward, one forward per block)."""
    cfg = _cfg_vocab(2)
    w = model.Weights(cfg)
    s = model.Session(cfg, w, max_seq=400); s.prefill([0] * 20)
    assert s.generate("selfspec-quad", 96, cands=(0, 3)) == [0] * 96
    assert s.forwards == 1 + 3 and s.accept_lens == [32, 32, 32]


def test_quadratic_candidate_draft_is_the_masked_draft_of_the_new_state():
    """After a cycle whose acceptance length L < 32 was a candidate, the draft
    it leaves is the masked draft computed afresh from the committed tokens
    (prefix length P + L + 1, the correction pending): the positions and the
    prefix of every candidate block are those of the state it stands for."""
    cfg = _cfg_vocab(8, seed=11)
    w = model.Weights(cfg)
    pr = [int(x) for x in synth.prompt(24, cfg.vocab, 5)]
    q = model.Session(cfg, w, max_seq=900); q.prefill(pr)
    checked = 0
    while len(q.tokens) < 200 and checked < 4:
        q.step_selfspec_quadratic(tuple(range(32)))
        if q.pending_draft is not None and q.accept_lens[-1] < 32:
            fresh = model.Session(cfg, w, max_seq=900)
            fresh.prefill(pr + q.tokens)
            assert fresh.kv_len == q.kv_len and fresh.last == q.last
            assert np.array_equal(fresh.draft_masked(), q.pending_draft)
            checked += 1
    assert checked >= 2
