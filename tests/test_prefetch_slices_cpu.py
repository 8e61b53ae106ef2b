"""Host-side check of the address arithmetic of the attention kernel's L2
prefetches (a plain Python model of it): the output projection's weights are
split into one slice per CTA, issued in bulk prefetches of at most 64 KB, and a
stream-K projection's runs are prefetched at k-steps [6, 12) past each run's
start. Every prefetched byte must lie inside the weight buffer, the first
prefetch must cover the buffer exactly once, and the second must stay inside
each run. The kernel only reads these addresses (a prefetch writes nothing),
but a range past the buffer would pull unrelated memory into L2."""
import pytest

CHUNK = 65536
KSTEP = 16384  # bytes of one 128 x 64 bf16 weight box in tiled storage


def _slices(total, nct):
    """(start, size) of every bulk prefetch, as the CTAs issue them."""
    total &= ~15
    per = ((total + nct - 1) // nct + CHUNK - 1) & ~(CHUNK - 1)
    out = []
    for cid in range(nct):
        b0 = per * cid
        b1 = min(b0 + per, total)
        o = b0
        while o < b1:
            n = min(b1 - o, CHUNK)
            out.append((o, n))
            o += CHUNK
    return out


def _runs(U, G, nct):
    out = []
    for cid in range(nct):
        for c in range(cid, G, nct):
            s0, s1 = c * U // G, (c + 1) * U // G
            k0, k1 = s0 + 6, min(s1, s0 + 12)
            if k1 > k0:
                out.append((c, s0, s1, k0, k1))
    return out


@pytest.mark.parametrize("total", [4096 * 4096 * 2, 1024 * 1024 * 2, 4096 * 4096 * 2 + 48, 12345 * 16])
@pytest.mark.parametrize("nct", [8, 64, 128, 136, 148, 4096])
def test_projection_prefetch_covers_the_buffer_once(total, nct):
    sl = _slices(total, nct)
    covered = 0
    last_end = 0
    for o, n in sorted(sl):
        assert o % 16 == 0 and n % 16 == 0 and 0 < n <= CHUNK
        assert o == last_end, "gap or overlap"
        assert o + n <= total
        last_end = o + n
        covered += n
    assert covered == total & ~15


@pytest.mark.parametrize("ntiles,nks", [(192, 64), (48, 64), (32, 64), (32, 192), (1187, 64)])
@pytest.mark.parametrize("nct", [8, 128, 136, 148])
def test_run_prefetch_stays_inside_each_run_and_the_buffer(ntiles, nks, nct):
    U = ntiles * nks
    G = min(148, U)
    runs = _runs(U, G, nct)
    seen = set()
    for c, s0, s1, k0, k1 in runs:
        assert s0 + 6 == k0 and k1 <= s1 and k1 <= U
        assert k1 * KSTEP <= U * KSTEP
        seen.add(c)
    # every run long enough gets its prefetch, from exactly one CTA
    assert seen == {c for c in range(G) if (c + 1) * U // G > c * U // G + 6}
    assert len(runs) == len(seen)
