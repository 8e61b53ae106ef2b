"""Host-side check of the lane arithmetic the large-batch unmask kernel uses
(four lanes per 32-slot sequence): a plain Python model of that arithmetic —
order-preserving integer keys, the lower-slot tie rule folded in as +1 on a
partner's key, the shuffles between the four lanes, and the merge of chosen
tokens into each lane's 16-byte chunks of the draft and next-input rows with
the shift by one crossing lanes — agrees with the oracle's unmask round on
random rows, tie-heavy rows, signed zeros, infinities and full masks. The GPU
kernel itself is checked against the oracle by the GPU parity tests."""
import numpy as np

from oracle import decode as OD


def _key(c):
    u = int(np.float32(c).view(np.uint32))
    if u == 0x80000000:
        u = 0
    return (~u & 0xFFFFFFFF) if u & 0x80000000 else (u | 0x80000000)


def _slot(q, e):
    return 4 * q + e if e < 4 else 16 + 4 * q + (e - 4)


def _lane_model(conf, pred, mask, k, block_in, draft):
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
        m, ch, bi, dr = _lane_model(conf, pred, mask, k, block_in, draft)
        rm, rb, rd, rch = OD.unmask(conf[None], pred[None], np.array([mask], np.uint32),
                                    block_in[None], draft[None], k)
        assert m == rm[0] and ch == list(rch[0]), trial
        assert np.array_equal(bi, rb[0]) and np.array_equal(dr, rd[0]), trial
