"""Pins of the oracle's logits reduction, unmask and verify/accept: brute force
with library sorts, library softmax, closed forms, exhaustive enumeration."""
import itertools

import numpy as np
import pytest
import torch

from oracle import decode as Dd


def _ref_reduce(row, excl):
    """Lowest-index argmax via a stable library sort; conf via torch.softmax."""
    keys = np.array(row, dtype=np.float64)
    order = np.argsort(-keys, kind="stable")
    order = [i for i in order if i != excl]
    if not order:
        return -1, 0.0
    best = int(order[0])
    p = torch.softmax(torch.from_numpy(keys), 0).numpy()
    return best, float(p[best])


@pytest.mark.parametrize("excl", [-1, 0, 17, 63])
def test_logits_reduce_vs_sort_and_softmax(excl):
    rng = np.random.default_rng(excl + 5)
    # bf16-like coarse values so ties are frequent
    x = np.round(rng.standard_normal((50, 64)) * 4) / 8
    ids, conf = Dd.logits_reduce(x, exclude_id=excl)
    for r in range(50):
        b, c = _ref_reduce(x[r], excl)
        assert ids[r] == b
        assert abs(conf[r] - c) <= 1e-14


def test_logits_reduce_closed_forms():
    V = 100
    x = np.zeros((3, V))
    x[1, 42] = np.log(7.0)          # one raised logit
    x[2, 0] = 5.0                   # excluded id holds the max
    ids, conf = Dd.logits_reduce(x, exclude_id=0)
    assert ids[0] == 1 and abs(conf[0] - 1 / V) < 1e-15          # all equal: lowest allowed id
    assert ids[1] == 42 and abs(conf[1] - 7 / (V - 1 + 7)) < 1e-15
    assert ids[2] == 1 and abs(conf[2] - 1 / (V - 1 + np.exp(5.0))) < 1e-15
    ids, conf = Dd.logits_reduce(np.zeros((1, 1)), exclude_id=0)  # nothing allowed
    assert ids[0] == -1 and conf[0] == 0.0


def _ref_unmask(conf_row, mask, k, T):
    masked = [i for i in range(T) if (mask >> i) & 1]
    # stable library sort on -conf keeps the lower slot first among ties
    order = [masked[j] for j in np.argsort(-np.asarray([conf_row[i] for i in masked]), kind="stable")]
    return order[:k]


@pytest.mark.parametrize("T", [1, 3, 6])
def test_unmask_exhaustive_small(T):
    rng = np.random.default_rng(T)
    for trial in range(3):
        conf = (rng.integers(1, 4, size=(1, T)) / 4.0)  # heavy ties
        pred = rng.integers(0, 1000, size=(1, T))
        for mask in range(1 << T):
            for k in range(1, T + 1):
                blk = np.full((1, T), 7, dtype=np.int32)
                dr = np.full((1, T), -1, dtype=np.int32)
                m2, b2, d2, ch = Dd.unmask(conf, pred, [mask], blk, dr, k)
                sel = _ref_unmask(conf[0], mask, k, T)
                assert list(ch[0, :len(sel)]) == sel
                assert all(c == -1 for c in ch[0, len(sel):])
                exp_mask = mask
                for i in sel:
                    exp_mask &= ~(1 << i)
                assert int(m2[0]) == exp_mask
                for i in range(T):
                    assert d2[0, i] == (pred[0, i] if i in sel else -1)
                    src = i - 1
                    assert b2[0, i] == (pred[0, src] if src in sel else 7)


def test_unmask_random_T32():
    rng = np.random.default_rng(11)
    B, T = 40, 32
    conf = rng.random((B, T))
    conf[::2] = np.round(conf[::2] * 8) / 8
    pred = rng.integers(0, 50000, size=(B, T))
    masks = rng.integers(0, 1 << 32, size=B)
    for k in (1, 4, 8, 32):
        m2, b2, d2, ch = Dd.unmask(conf, pred, masks, np.zeros((B, T)), np.full((B, T), -1), k)
        for b in range(B):
            sel = _ref_unmask(conf[b], int(masks[b]), k, T)
            assert list(ch[b, :len(sel)]) == sel
            assert bin(int(m2[b])).count("1") == bin(int(masks[b])).count("1") - len(sel)


def test_verify_accept_bruteforce():
    rng = np.random.default_rng(3)
    B, T = 200, 32
    target = rng.integers(0, 5, size=(B, T))
    draft = np.where(rng.random((B, T)) < 0.9, target, rng.integers(0, 5, size=(B, T)))
    draft[0] = target[0]
    kv = rng.integers(0, 100, size=B)
    L, commit, n, kv2 = Dd.verify_accept(draft, target, kv)
    eq = (draft == target).astype(np.int64)
    Lref = np.cumprod(eq, axis=1).sum(axis=1)
    assert np.array_equal(L, Lref)
    assert L[0] == T and n[0] == T
    assert np.array_equal(n, np.minimum(Lref + 1, T))
    assert np.array_equal(kv2, kv + n)
    for b in range(B):
        assert list(commit[b, :n[b]]) == list(target[b, :n[b]])
        assert (commit[b, n[b]:] == -1).all()
        if L[b] < T:
            assert commit[b, L[b]] == target[b, L[b]] and draft[b, L[b]] != target[b, L[b]]


# ---------------------------------------------------------------- threshold sampler
def _round(conf, pred, mask, tau, tau_rev=2.0, T=None, draft=None):
    conf = np.asarray(conf, dtype=np.float64)[None]
    T = conf.shape[1]
    blk = np.full((1, T), 7, dtype=np.int32)
    dr = np.full((1, T), -1, dtype=np.int32) if draft is None else np.asarray(draft)[None].astype(np.int32)
    return Dd.unmask_threshold(conf, np.asarray(pred)[None], [mask], blk, dr, tau, tau_rev)


@pytest.mark.parametrize("T", [1, 4, 6])
def test_threshold_above_one_is_the_top1_rule(T):
    """tau > 1 (no confidence reaches it) fixes exactly the slot the fixed-k
    rule with k = 1 fixes, for every mask."""
    rng = np.random.default_rng(20 + T)
    conf = rng.integers(1, 4, size=(1, T)) / 4.0
    pred = rng.integers(0, 1000, size=(1, T))
    for mask in range(1, 1 << T):
        blk = np.full((1, T), 7, dtype=np.int32)
        dr = np.full((1, T), -1, dtype=np.int32)
        a = Dd.unmask(conf, pred, [mask], blk, dr, 1)
        b = Dd.unmask_threshold(conf, pred, [mask], blk, dr, 1.5)
        assert int(a[0][0]) == int(b[0][0]) and np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
        assert b[3][0] == 1


@pytest.mark.parametrize("T", [1, 5, 32])
def test_threshold_at_zero_fixes_every_masked_slot(T):
    """tau <= min conf fixes all masked slots at once: the fixed-k rule with k = T."""
    rng = np.random.default_rng(30 + T)
    conf = rng.random((1, T)) + 1e-3
    pred = rng.integers(0, 1000, size=(1, T))
    mask = int(rng.integers(1, 1 << T))
    blk = np.full((1, T), 7, dtype=np.int32)
    dr = np.full((1, T), -1, dtype=np.int32)
    a = Dd.unmask(conf, pred, [mask], blk, dr, T)
    b = Dd.unmask_threshold(conf, pred, [mask], blk, dr, 0.0)
    assert int(b[0][0]) == 0 and np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    assert b[3][0] == bin(mask).count("1")


def test_threshold_counts_and_inputs_bruteforce():
    """Random rounds: the fixed set is {masked, conf >= tau} or the first
    maximiser; block_in[i+1] carries draft[i] for every fixed slot."""
    rng = np.random.default_rng(41)
    T = 32
    for trial in range(300):
        conf = np.round(rng.random(T) * 8) / 8
        pred = rng.integers(0, 100, size=T)
        mask = int(rng.integers(0, 1 << T))
        tau = float(rng.choice([0.25, 0.5, 0.875, 1.0, 1.5]))
        m2, b2, d2, nf, nr = _round(conf, pred, mask, tau)
        masked = [i for i in range(T) if (mask >> i) & 1]
        want = [i for i in masked if conf[i] >= tau]
        if not want and masked:
            top = max(conf[i] for i in masked)
            want = [min(i for i in masked if conf[i] == top)]
        assert nf[0] == len(want) and nr[0] == 0
        assert int(m2[0]) == mask & ~sum(1 << i for i in want)
        for i in range(T):
            assert d2[0, i] == (pred[i] if i in want else -1)
            if i >= 1:
                assert b2[0, i] == (pred[i - 1] if i - 1 in want else 7)


def test_revision_replaces_disagreeing_earlier_slots():
    """Slots fixed in earlier rounds are replaced exactly when the new
    prediction differs and its confidence reaches tau_revise; slots fixed
    in this round are not revised; tau_revise > 1 never revises."""
    T = 8
    draft = np.array([5, 6, 7, 8, -1, -1, -1, -1])
    pred = np.array([5, 60, 70, 80, 1, 2, 3, 4])
    conf = np.array([0.9, 0.9, 0.3, 0.6, 0.1, 0.95, 0.2, 0.2])
    mask = 0b11110000
    m2, b2, d2, nf, nr = _round(conf, pred, mask, 0.9, 0.5, draft=draft)
    assert nr[0] == 2                       # slots 1 (0.9) and 3 (0.6); slot 2 below 0.5; slot 0 agrees
    assert list(d2[0, :4]) == [5, 60, 7, 80]
    assert b2[0, 2] == 60 and b2[0, 4] == 80 and b2[0, 3] == 7
    assert nf[0] == 1 and d2[0, 5] == 2 and int(m2[0]) == 0b11010000
    m3, b3, d3, nf3, nr3 = _round(conf, pred, mask, 0.9, 1.5, draft=draft)
    assert nr3[0] == 0 and list(d3[0, :4]) == [5, 6, 7, 8]
