"""Pins of the oracle's Philox4x64-10 (numpy's independent implementation and
the generator's published known-answer vector), its Box-Muller stream (closed
forms, moments) and its bf16 rounding (torch's conversion)."""
import numpy as np
import torch

from oracle import numerics, philox


def test_philox_known_answer():
    # Known-answer vector of Philox4x64-10 for zero counter and zero key, as
    # distributed with the generator's reference implementation (Random123).
    got = philox.philox4x64_10(0, 0, 0, 0, 0, 0)
    assert [int(x) for x in got] == [0x16554D9ECA36314C, 0xDB20FE9D672D0FDC,
                                     0xD7E772CEE186176B, 0x7E68B68AEC7BA23B]


def test_philox_matches_numpy_bit_generator():
    # numpy.random.Philox increments its 256-bit counter before each block.
    rng = np.random.default_rng(0)
    for _ in range(20):
        key = [int(x) for x in rng.integers(0, 2**63, size=2)]
        ctr = [int(x) for x in rng.integers(0, 2**63, size=2)]
        bg = np.random.Philox(key=key, counter=[ctr[0], ctr[1], 0, 0])
        ref = bg.random_raw(8)
        got0 = philox.philox4x64_10(ctr[0] + 1, ctr[1], 0, 0, key[0], key[1])
        got1 = philox.philox4x64_10(ctr[0] + 2, ctr[1], 0, 0, key[0], key[1])
        assert [int(x) for x in got0] + [int(x) for x in got1] == [int(x) for x in ref]


def test_raw_blocks_equal_the_definition():
    """The bulk generator (NumPy's C Philox started one block early) gives the
    same words as the pure-NumPy definition, including the counter edges
    (block 0 of tensor 0 and of tensor 5)."""
    for seed, tid, n0, nb in ((0, 0, 0, 7), (1005, 5, 0, 3), (77, 9, 12345, 11), (3, 0, 2**40, 4)):
        got = philox.raw_blocks(seed, tid, n0, nb)
        n = np.arange(n0, n0 + nb, dtype=np.uint64)
        ref = philox.philox4x64_10(n, np.uint64(tid), np.uint64(0), np.uint64(0),
                                   np.uint64(seed), np.uint64(0))
        for a, b in zip(got, ref):
            assert np.array_equal(a, b)


def test_box_muller_closed_forms():
    top = np.uint64((2**53 - 1) << 11)   # u1 = 1 -> r = 0
    z0, z1 = philox.box_muller(np.array([top]), np.array([np.uint64(0)]))
    assert z0[0] == 0.0 and z1[0] == 0.0
    w = np.uint64((2**52 - 1) << 11)     # u1 = 1/2
    z0, z1 = philox.box_muller(np.array([w]), np.array([np.uint64(0)]))
    assert abs(z0[0] - np.sqrt(2 * np.log(2))) < 1e-15 and z1[0] == 0.0
    quarter = np.uint64(2**51 << 11)     # u2 = 1/4 -> theta = pi/2
    z0, z1 = philox.box_muller(np.array([w]), np.array([quarter]))
    assert abs(z0[0]) < 1e-15 and abs(z1[0] - np.sqrt(2 * np.log(2))) < 1e-15


def test_normal_stream_moments_and_random_access():
    n = 1_000_000
    z = philox.normal_stream(7, 3, 0, n)
    se = 1 / np.sqrt(n)
    assert abs(z.mean()) < 4 * se
    assert abs(z.var() - 1) < 4 * np.sqrt(2) * se
    assert abs((z ** 4).mean() - 3) < 4 * np.sqrt(96) * se
    # any window of the stream can be drawn on its own
    assert np.array_equal(philox.normal_stream(7, 3, 12345, 77), z[12345:12345 + 77])
    # different tensors are different streams
    assert not np.array_equal(philox.normal_stream(7, 4, 0, 16), z[:16])


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10,
                        np.array([1.00390625, 1.01171875, -1.00390625, 3.0e38, 1e-40, 0.0, -0.0],
                                 dtype=np.float32)])
    # exact ties between two bf16 neighbours
    ties = ((rng.integers(0, 1 << 16, 1000).astype(np.uint32) << 16) | 0x8000).view(np.float32)
    x = np.concatenate([x, ties[np.isfinite(ties)]])
    ours = numerics.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_f64_to_bf16_is_correctly_rounded():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(200000) * 3
    got = numerics.round_to_bf16(x)
    # brute force: among the bf16 grid points around x pick the nearer (even on ties)
    for xi, gi in zip(x[:2000], got[:2000]):
        cands = []
        b = (np.array([xi], dtype=np.float32).view(np.uint32)[0] >> 16)
        for d in (-1, 0, 1, 2):
            c = float(numerics.bf16_bits_to_f64(np.array([(int(b) + d) & 0xFFFF], dtype=np.uint16))[0])
            cands.append(c)
        best = min(cands, key=lambda c: (abs(c - xi), (np.array([c], dtype=np.float32).view(np.uint32)[0] >> 16) & 1))
        assert gi == best
