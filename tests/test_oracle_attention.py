"""Pins of the oracle's block-causal attention against facts fixed outside it:
torch's scaled_dot_product_attention (a library routine) with independently
built masks, closed forms, and the invariants the definition implies."""
import numpy as np
import pytest
import torch

from oracle import attention as A


def _rand(B, T, Hq, Hkv, D, P, seed, Lmax=None):
    rng = np.random.default_rng(seed)
    Lmax = Lmax or (max(np.atleast_1d(P)) + T + 3)
    q = rng.standard_normal((B, T, Hq, D))
    k = rng.standard_normal((B, Hkv, Lmax, D))
    v = rng.standard_normal((B, Hkv, Lmax, D))
    kv = np.broadcast_to(np.atleast_1d(P), (B,)).astype(np.int64)
    return q, k, v, kv


def _sdpa(q, k, v, mask=None, scale=None):
    """torch SDPA in float64; q [H][Tq][D], k/v [H][Tk][D], mask [Tq][Tk] bool."""
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
        attn_mask=None if mask is None else torch.from_numpy(mask), scale=scale).numpy()


@pytest.mark.parametrize("T", [1, 5, 32])
def test_empty_prefix_bidir_is_full_attention(T):
    q, k, v, kv = _rand(1, T, 4, 4, 16, 0, 1)
    out = A.block_attn(q, k, v, kv, A.BIDIR, 0.25)
    ref = _sdpa(q[0].transpose(1, 0, 2), k[0, :, :T], v[0, :, :T], scale=0.25).transpose(1, 0, 2)
    np.testing.assert_allclose(out[0], ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("P,T", [(0, 7), (5, 7), (40, 32), (3, 1)])
def test_causal_block_matches_masked_sdpa(P, T):
    q, k, v, kv = _rand(1, T, 2, 2, 8, P, 2)
    scale = 1 / np.sqrt(8)
    out = A.block_attn(q, k, v, kv, A.CAUSAL, scale)
    # query slot i sits at position P+i and may see keys 0..P+i
    mask = np.tril(np.ones((T, P + T), dtype=bool), k=P)
    ref = _sdpa(q[0].transpose(1, 0, 2), k[0, :, :P + T], v[0, :, :P + T], mask, scale)
    np.testing.assert_allclose(out[0], ref.transpose(1, 0, 2), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("P", [0, 9])
def test_bidir_block_sees_prefix_and_whole_block(P):
    T = 6
    q, k, v, kv = _rand(1, T, 2, 1, 8, P, 3)
    out = A.block_attn(q, k, v, kv, A.BIDIR, 0.3)
    ref = _sdpa(q[0].transpose(1, 0, 2), np.repeat(k[0, :, :P + T], 2, 0),
                np.repeat(v[0, :, :P + T], 2, 0), None, 0.3)
    np.testing.assert_allclose(out[0], ref.transpose(1, 0, 2), rtol=1e-12, atol=1e-12)


def test_block_size_one_is_causal_decode():
    q, k, v, kv = _rand(2, 1, 4, 2, 8, [11, 4], 4)
    a = A.block_attn(q, k, v, kv, A.BIDIR, 0.5)
    c = A.block_attn(q, k, v, kv, A.CAUSAL, 0.5)
    assert np.array_equal(a, c)
    for b, P in enumerate([11, 4]):
        ref = _sdpa(q[b].transpose(1, 0, 2), np.repeat(k[b, :, :P + 1], 2, 0),
                    np.repeat(v[b, :, :P + 1], 2, 0), None, 0.5)
        np.testing.assert_allclose(a[b], ref.transpose(1, 0, 2), rtol=1e-12, atol=1e-12)


def test_causal_rows_equal_single_token_calls():
    """Slot i of a CAUSAL block equals a T=1 call whose prefix holds the earlier
    block keys: bit-exact, the property that makes self-speculation equal AR."""
    P, T = 13, 9
    q, k, v, kv = _rand(1, T, 4, 2, 16, P, 5)
    blk = A.block_attn(q, k, v, kv, A.CAUSAL, 0.25)
    for i in range(T):
        one = A.block_attn(q[:, i:i + 1], k, v, np.array([P + i]), A.CAUSAL, 0.25)
        assert np.array_equal(one[0, 0], blk[0, i])


def test_bidir_permutation_equivariance():
    P, T = 7, 8
    q, k, v, kv = _rand(1, T, 2, 2, 8, P, 6)
    out = A.block_attn(q, k, v, kv, A.BIDIR, 0.4)
    perm = np.random.default_rng(0).permutation(T)
    # permuting the queries permutes the outputs
    out_q = A.block_attn(q[:, perm], k, v, kv, A.BIDIR, 0.4)
    np.testing.assert_allclose(out_q, out[:, perm], rtol=1e-13, atol=1e-13)
    # permuting the block keys together with their values changes nothing
    k2, v2 = k.copy(), v.copy()
    k2[:, :, P:P + T] = k[:, :, P + perm]
    v2[:, :, P:P + T] = v[:, :, P + perm]
    np.testing.assert_allclose(A.block_attn(q, k2, v2, kv, A.BIDIR, 0.4), out, rtol=1e-12, atol=1e-13)


def test_gqa_equals_mha_with_replicated_kv():
    P, T, G = 10, 4, 4
    q, k, v, kv = _rand(2, T, 8, 2, 8, [P, P + 3], 7)
    gqa = A.block_attn(q, k, v, kv, A.CAUSAL, 0.3)
    mha = A.block_attn(q, np.repeat(k, G, 1), np.repeat(v, G, 1), kv, A.CAUSAL, 0.3)
    assert np.array_equal(gqa, mha)


def test_closed_forms():
    P, T, D = 5, 3, 8
    q, k, v, kv = _rand(1, T, 2, 2, D, P, 8)
    # constant value rows: output is that constant whatever the weights (rows sum to 1)
    vc = np.ones_like(v) * 2.5
    out = A.block_attn(q, k, vc, kv, A.CAUSAL, 0.7)
    np.testing.assert_allclose(out, 2.5, rtol=0, atol=1e-13)
    # zero query: uniform weights, output is the mean of the visible value rows
    out = A.block_attn(np.zeros_like(q), k, v, kv, A.CAUSAL, 0.7)
    for i in range(T):
        np.testing.assert_allclose(out[0, i, 0], v[0, 0, :P + i + 1].mean(0), rtol=1e-12, atol=1e-13)
    # a single visible key: the output is its value row
    out = A.block_attn(q[:, :1], k, v, np.array([0]), A.CAUSAL, 0.7)
    np.testing.assert_allclose(out[0, 0, 1], v[0, 1, 0], rtol=0, atol=0)


def test_scale_and_sign_matter():
    """Two keys: the weight on key 1 is sigmoid(scale*(s1-s0)) exactly."""
    q = np.zeros((1, 1, 1, 2)); q[0, 0, 0] = [1.0, 0.0]
    k = np.zeros((1, 1, 2, 2)); k[0, 0, 0] = [0.0, 0.0]; k[0, 0, 1] = [3.0, 0.0]
    v = np.zeros((1, 1, 2, 2)); v[0, 0, 0] = [1.0, 0.0]; v[0, 0, 1] = [0.0, 1.0]
    out = A.block_attn(q, k, v, np.array([1]), A.CAUSAL, 0.5)
    w1 = 1 / (1 + np.exp(-1.5))
    np.testing.assert_allclose(out[0, 0, 0], [1 - w1, w1], rtol=1e-14)


def test_rows_helper_matches_full():
    q, k, v, kv = _rand(2, 5, 4, 2, 8, [6, 2], 9)
    full = A.block_attn(q, k, v, kv, A.CAUSAL, 0.3)
    rows = [(0, 0, 0), (1, 4, 3), (0, 2, 1)]
    got = A.block_attn_rows(q, k, v, kv, A.CAUSAL, 0.3, rows)
    for r, (b, i, h) in enumerate(rows):
        assert np.array_equal(got[r], full[b, i, h])
