"""Host-side check of the stream-K bookkeeping the projection kernel and its
consumers share (a plain Python model of the integer arithmetic): CTA c of G
owns the k-steps [c U / G, (c + 1) U / G) of the U = tiles x nks k-steps, in
tile-major order, and leaves one partial tile per segment (the part of one
tile it covers).

- With the deferred merge (GEMM_EPI_PARTIAL) segment s of CTA c goes to slot
  c * maxseg + s, and a consumer finds tile t's contributors as
  cf = ((t nks + 1) G - 1) / U .. cl = ((t nks + nks) G - 1) / U and
  contributor c's slot for t as t - (c U / G) / nks.
- With the in-kernel merge each CTA keeps at most two partials: slot 1 for the
  segment that starts at a tile's first k-step, slot 0 for one that starts
  inside a tile; the merger reads cf's slot 1 and every later contributor's
  slot 0.

The model checks that both views agree with a brute-force walk of every CTA's
run, that maxseg bounds the segments, and that the in-kernel merge's two slots
never collide, over the 8B projections and random shapes and grid sizes."""
import random

import pytest


def _segments(c, U, G, nks):
    """(tile, first k-step in the tile, last k-step + 1) of CTA c's run, in order."""
    kb0, kb1 = c * U // G, (c + 1) * U // G
    out = []
    g = kb0
    while g < kb1:
        tile, lo = g // nks, g % nks
        hi = min(nks, lo + (kb1 - g))
        out.append((tile, lo, hi))
        g += hi - lo
    return out


def _maxseg(U, G, nks):
    run = (U + G - 1) // G
    return (run + nks - 1) // nks + 1


def _check(ntiles, nks, G):
    U = ntiles * nks
    G = min(G, U)
    maxseg = _maxseg(U, G, nks)
    contrib = {t: [] for t in range(ntiles)}
    for c in range(G):
        segs = _segments(c, U, G, nks)
        assert len(segs) <= maxseg
        for s, (tile, lo, hi) in enumerate(segs):
            contrib[tile].append((c, s, lo, hi))
        # in-kernel merge: at most one partial in each of the two slots
        partial = [(lo > 0) for (tile, lo, hi) in segs if not (lo == 0 and hi == nks)]
        assert partial.count(True) <= 1 and partial.count(False) <= 1, (c, segs)
    for t in range(ntiles):
        cs = contrib[t]
        # the k-steps of the tile are covered exactly once, in contributor order
        assert [lo for _, _, lo, _ in cs][0] == 0 and cs[-1][3] == nks
        for (a, _, _, ahi), (b, _, blo, _) in zip(cs, cs[1:]):
            assert b == a + 1 and blo == ahi
        t0 = t * nks
        cf = ((t0 + 1) * G - 1) // U
        cl = ((t0 + nks) * G - 1) // U
        assert (cf, cl) == (cs[0][0], cs[-1][0]), (t, cf, cl, cs)
        for c, s, lo, hi in cs:
            assert t - (c * U // G) // nks == s  # the consumer's slot rule
            if len(cs) > 1:  # split tile: the in-kernel merge's slot rule
                my_slot = 0 if lo > 0 else 1
                assert my_slot == (1 if c == cf else 0)


@pytest.mark.parametrize("ntiles,nks", [(48, 64), (32, 64), (192, 64), (32, 192), (1187, 64), (2, 4), (1, 64)])
@pytest.mark.parametrize("G", [1, 7, 96, 148, 160])
def test_streamk_bookkeeping_8b_shapes(ntiles, nks, G):
    _check(ntiles, nks, G)


def test_streamk_bookkeeping_random_shapes():
    rng = random.Random(5)
    for _ in range(400):
        _check(rng.randint(1, 300), rng.randint(1, 200), rng.randint(1, 200))
