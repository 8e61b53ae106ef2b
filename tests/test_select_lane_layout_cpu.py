"""Host-side check of the lane arithmetic the large-batch unmask kernel uses
(four lanes per 32-slot sequence): a plain Python model of that arithmetic —
order-preserving integer keys, the lower-slot tie rule folded in as +1 on a
partner's key, the shuffles between the four lanes, and the merge of chosen
tokens into each lane's 16-byte chunks of the draft and next-input rows with
the shift by one crossing lanes — agrees with the oracle's unmask round on
random rows, tie-heavy rows, signed zeros, infinities and full masks. The GPU
kernel itself is checked against the oracle by the GPU parity tests. For
k <= 8 the kernel takes the winners by extraction instead of ranking every
slot (a sorting network per lane, then the largest of the four lanes' heads
per round); the model of that path must give the same result."""
import numpy as np

from oracle import decode as OD


def _key(c):
    u = int(np.float32(c).view(np.uint32))
    if u == 0x80000000:
        u = 0
    return (~u & 0xFFFFFFFF) if u & 0x80000000 else (u | 0x80000000)


def _slot(q, e):
    return 4 * q + e if e < 4 else 16 + 4 * q + (e - 4)


# the 19-comparator sorting network of the extraction path (descending)
_NET = [(0, 1), (2, 3), (4, 5), (6, 7), (0, 2), (1, 3), (4, 6), (5, 7), (1, 2), (5, 6),
        (0, 4), (1, 5), (2, 6), (3, 7), (2, 4), (3, 5), (1, 2), (3, 4), (5, 6)]


def _extract_ranks(key, mask, k):
    """The k <= 8 path: each lane sorts its composite keys (key << 5 | 31 - slot)
    with the network; round r takes the largest of the four lanes' heads."""
    kk = min(k, bin(mask).count("1"))
    lists = []
    for q in range(4):
        sk = [(key[q][e] << 5) | (31 - _slot(q, e)) for e in range(8)]
        for a, b in _NET:
            if sk[b] > sk[a]:
                sk[a], sk[b] = sk[b], sk[a]
        lists.append(sk)
    rank = [[99] * 8 for _ in range(4)]
    for r in range(k):
        heads = [lst[0] for lst in lists]
        m = max(max(heads[0], heads[1]), max(heads[2], heads[3]))
        if r < kk:
            q = heads.index(m)
            slot = 31 - (m & 31)
            e = next(e for e in range(8) if _slot(q, e) == slot)
            rank[q][e] = r
            lists[q] = lists[q][1:] + [0]
    return rank


def _lane_model(conf, pred, mask, k, block_in, draft, extract=False):
    key = [[_key(conf[_slot(q, e)]) if (mask >> _slot(q, e)) & 1 else 0 for e in range(8)]
           for q in range(4)]
    rank = [[0] * 8 for _ in range(4)]
    for q in range(4):
        for e in range(8):
            for f in range(e + 1, 8):
                p = int(key[q][f] > key[q][e])
                rank[q][e] += p
                rank[q][f] += 1 - p
        for d in (1, 2, 3):
            o = key[q ^ d]
            lower = int((q ^ d) < q)
            for f in range(8):
                for e in range(8):
                    # partner slot below own slot: same half and lower lane, or
                    # partner in the first half and own in the second
                    if f < 4:
                        adj = lower if e < 4 else 1
                    else:
                        adj = 0 if e < 4 else lower
                    rank[q][e] += int(o[f] + adj > key[q][e])
    kk = min(k, bin(mask).count("1"))
    if extract:
        rank = _extract_ranks(key, mask, k)
    sel = [[key[q][e] != 0 and rank[q][e] < kk for e in range(8)] for q in range(4)]
    chosen = [-1] * k
    taken = 0
    new_draft, new_in = draft.copy(), block_in.copy()
    for q in range(4):
        src = (q + 3) & 3  # the lower lane, lane 3 for lane 0
        carry_first = q > 0 and sel[src][3]
        carry_second = sel[src][7] if q > 0 else sel[src][3]
        carry_second_val = pred[_slot(src, 7)] if q > 0 else pred[_slot(src, 3)]
        for e in range(8):
            if sel[q][e]:
                i = _slot(q, e)
                new_draft[i] = pred[i]
                chosen[rank[q][e]] = i
                taken |= 1 << i
        firsts = [(carry_first, pred[_slot(src, 3)])] + [(sel[q][e], pred[_slot(q, e)]) for e in range(3)]
        seconds = [(carry_second, carry_second_val)] + [(sel[q][e], pred[_slot(q, e)]) for e in range(4, 7)]
        for j in range(4):
            if firsts[j][0]:
                new_in[4 * q + j] = firsts[j][1]
            if seconds[j][0]:
                new_in[16 + 4 * q + j] = seconds[j][1]
    return mask & ~taken & 0xFFFFFFFF, chosen, new_in, new_draft


def test_lane_model_matches_oracle_unmask():
    rng = np.random.default_rng(12)
    special = np.array([0.0, -0.0, -np.inf, np.inf, 1e-30, -1e-30, 0.5, -0.5], dtype=np.float32)
    for trial in range(600):
        kind = trial % 3
        if kind == 0:
            conf = rng.random(32, dtype=np.float32)
        elif kind == 1:
            conf = (rng.integers(1, 5, 32) / 4).astype(np.float32)
        else:
            conf = special[rng.integers(0, len(special), 32)]
        pred = rng.integers(0, 1000, 32).astype(np.int32)
        mask = 0xFFFFFFFF if trial % 7 == 0 else int(rng.integers(0, 2**32))
        k = int(rng.integers(1, 33))
        block_in = rng.integers(-5, 0, 32).astype(np.int32)
        draft = rng.integers(-9, -5, 32).astype(np.int32)
        rm, rb, rd, rch = OD.unmask(conf[None], pred[None], np.array([mask], np.uint32),
                                    block_in[None], draft[None], k)
        for extract in ((False, True) if k <= 8 else (False,)):
            m, ch, bi, dr = _lane_model(conf, pred, mask, k, block_in, draft, extract)
            assert m == rm[0] and ch == list(rch[0]), (trial, extract)
            assert np.array_equal(bi, rb[0]) and np.array_equal(dr, rd[0]), (trial, extract)


def test_extraction_network_sorts_every_zero_one_input():
    """The network sorts (0-1 principle: every 0/1 input of length 8 suffices)."""
    import itertools
    for bits in itertools.product([0, 1], repeat=8):
        s = list(bits)
        for a, b in _NET:
            if s[b] > s[a]:
                s[a], s[b] = s[b], s[a]
        assert s == sorted(bits, reverse=True), bits
