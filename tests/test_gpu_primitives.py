"""GPU parity of the decode-step primitives against the oracle, through the C ABI.

Bars (stated by the workload's specification): integer outputs bit-exact;
attention |err| <= 1e-2 + 1e-2 |ref| (bf16 inputs, fp32 accumulation);
confidence relative error <= 1e-4."""
import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import decode as OD
from self_speculative_lm_block_b300 import synth

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-2, 1e-2


@pytest.fixture(scope="module")
def nd(cuda_ok):
    from self_speculative_lm_block_b300 import ndiff
    return ndiff


def _attn_check(nd, B, T, Hq, Hkv, D, lengths, Lmax, mode, seed, split=0, dtype=torch.bfloat16,
                fill=float("nan"), rows=None):
    inp = synth.attn_inputs(B, T, Hq, Hkv, D, lengths, Lmax, seed, dtype=dtype, fill_tail=fill)
    dev = "cuda"
    out = nd.block_attn(inp.q.to(dev), inp.k_cache.to(dev), inp.v_cache.to(dev),
                        inp.kv_len.to(dev), mode, inp.scale, split_keys=split)
    nd.ndiff_check()
    got = out.float().cpu().numpy()
    q = inp.q.float().numpy()
    k = inp.k_cache.float().numpy()
    v = inp.v_cache.float().numpy()
    if rows is None:
        ref = OA.block_attn(q, k, v, inp.kv_len.numpy(), mode, inp.scale)
        g = got
    else:
        ref = OA.block_attn_rows(q, k, v, inp.kv_len.numpy(), mode, inp.scale, rows)
        g = np.stack([got[b, i, h] for (b, i, h) in rows])
    err = np.abs(g - ref)
    tol = ATOL + RTOL * np.abs(ref)
    assert np.isfinite(g).all()
    assert (err <= tol).all(), f"max err {err.max():.3e} (worst excess {(err - tol).max():.3e})"
    return got


# ---------------------------------------------------------------- attention
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("T,lengths", [(32, [0, 70, 200]), (5, [1, 63, 64]), (1, [0, 129, 65])])
def test_attn_bf16_small(nd, mode, T, lengths):
    Lmax = max(lengths) + T + 37
    _attn_check(nd, len(lengths), T, 32, 8, 128, lengths, Lmax, mode, seed=11 + T)


@pytest.mark.parametrize("split", [64, 128, 256])
def test_attn_bf16_splits(nd, split):
    lengths = [300, 17, 511]
    _attn_check(nd, 3, 32, 32, 8, 128, lengths, 600, 1, seed=21, split=split)


@pytest.mark.parametrize("mode", [0, 1])
def test_attn_bf16_many_ragged_sequences(nd, mode):
    """Forty sequences with ragged prefixes (including empty and full caches),
    every row checked; the automatic schedule and an explicit 128-key split
    agree."""
    B, T, Lmax = 40, 32, 544
    lengths = np.random.default_rng(7).integers(0, Lmax - T + 1, size=B)
    lengths[:3] = [0, Lmax - T, 63]
    got = _attn_check(nd, B, T, 32, 8, 128, lengths, Lmax, mode, seed=33)
    # the same launch with an explicit split grid agrees within the bound
    inp = synth.attn_inputs(B, T, 32, 8, 128, lengths, Lmax, 33, fill_tail=float("nan"))
    alt = nd.block_attn(inp.q.cuda(), inp.k_cache.cuda(), inp.v_cache.cuda(), inp.kv_len.cuda(),
                        mode, inp.scale, split_keys=128).float().cpu().numpy()
    assert np.abs(got - alt).max() <= 2e-2


@pytest.mark.parametrize("split", [128, 1408])
def test_attn_bf16_batch_equals_single_sequences(nd, split):
    """A batch is launched longest item first; every sequence's rows are the
    same bits as a launch of that sequence alone with the same split grid."""
    B, T, Lmax = 6, 32, 1400
    lengths = [0, 5, 100, 1368, 700, 64]
    inp = synth.attn_inputs(B, T, 32, 8, 128, lengths, Lmax, 43, fill_tail=float("nan"))
    q, k, v = inp.q.cuda(), inp.k_cache.cuda(), inp.v_cache.cuda()
    both = nd.block_attn(q, k, v, inp.kv_len.cuda(), 1, inp.scale, split_keys=split)
    for b in range(B):
        one = nd.block_attn(q[b:b + 1].contiguous(), k[b:b + 1].contiguous(),
                            v[b:b + 1].contiguous(), inp.kv_len[b:b + 1].cuda(), 1, inp.scale,
                            split_keys=split)
        assert torch.equal(one[0], both[b]), b


def test_attn_bf16_gqa_group_2_and_mha(nd):
    _attn_check(nd, 2, 32, 16, 8, 128, [100, 40], 200, 0, seed=31)      # G = 2
    _attn_check(nd, 2, 16, 8, 1, 128, [100, 40], 200, 1, seed=32)       # G = 8, T = 16


def test_attn_bf16_single_8b_shape(nd):
    c = synth.ATTN_SINGLE
    for mode in (0, 1):
        _attn_check(nd, c["B"], c["T"], c["Hq"], c["Hkv"], c["D"], [c["P_lo"]], c["P_lo"] + c["T"],
                    mode, seed=c["seed"], fill=0.0)


def test_attn_bf16_batched_sampled_rows(nd):
    c = synth.ATTN_BATCHED
    lengths = synth.attn_lengths(c["B"], c["seed"], c["P_lo"], c["P_hi"])
    Lmax = c["P_hi"] + c["T"]
    rng = np.random.default_rng(0)
    rows = [(int(b), int(i), int(h)) for b, i, h in zip(rng.integers(0, c["B"], 200),
                                                        rng.integers(0, c["T"], 200),
                                                        rng.integers(0, c["Hq"], 200))]
    _attn_check(nd, c["B"], c["T"], c["Hq"], c["Hkv"], c["D"], lengths, Lmax, 1, seed=c["seed"],
                fill=0.0, rows=rows)


def test_attn_bf16_long_sampled_rows(nd):
    c = synth.ATTN_LONG
    rng = np.random.default_rng(1)
    rows = [(int(b), int(i), int(h)) for b, i, h in zip(rng.integers(0, c["B"], 64),
                                                        rng.integers(0, c["T"], 64),
                                                        rng.integers(0, c["Hq"], 64))]
    _attn_check(nd, c["B"], c["T"], c["Hq"], c["Hkv"], c["D"], [c["P_lo"]] * c["B"],
                c["P_lo"] + c["T"], 0, seed=c["seed"], fill=0.0, rows=rows)


def test_attn_bf16_rows_independent_of_block_length(nd):
    """A CAUSAL block of T rows equals T single-row calls at prefix P+i, bit for bit."""
    P, T = 700, 32
    inp = synth.attn_inputs(1, T, 32, 8, 128, [P], P + T + 64, 41, fill_tail=0.0)
    q, k, v = inp.q.cuda(), inp.k_cache.cuda(), inp.v_cache.cuda()
    blk = nd.block_attn(q, k, v, inp.kv_len.cuda(), 1, inp.scale)
    for i in range(T):
        one = nd.block_attn(q[:, i:i + 1].contiguous(), k, v,
                            torch.tensor([P + i], dtype=torch.int32, device="cuda"), 1, inp.scale)
        assert torch.equal(one[0, 0], blk[0, i]), i


@pytest.mark.parametrize("mode", [0, 1])
def test_attn_f32_tiny(nd, mode):
    for T, lengths in ((32, [0, 45]), (1, [31, 7]), (9, [3, 80])):
        Lmax = max(lengths) + T + 5
        inp = synth.attn_inputs(2, T, 4, 4, 32, lengths, Lmax, 51, dtype=torch.float32,
                                fill_tail=float("nan"))
        out = nd.block_attn(inp.q.cuda(), inp.k_cache.cuda(), inp.v_cache.cuda(),
                            inp.kv_len.cuda(), mode, inp.scale)
        ref = OA.block_attn(inp.q.numpy(), inp.k_cache.numpy(), inp.v_cache.numpy(),
                            inp.kv_len.numpy(), mode, inp.scale)
        np.testing.assert_allclose(out.cpu().numpy(), ref, rtol=1e-5, atol=1e-5)


def test_attn_rejects_bad_shapes(nd):
    q = torch.zeros((1, 32, 32, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 8, 64, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(nd.NdiffError) as e:
        nd.block_attn(q, k, k, torch.zeros(1, dtype=torch.int32, device="cuda"), 0, 0.1)
    assert e.value.status == nd.NDIFF_ERR_UNSUPPORTED


# ---------------------------------------------------------------- logits reduce
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("V,ld,excl", [(1003, 1008, 5), (512, 512, 511), (8, 8, -1), (1, 8, 0),
                                       (37, 40, 36)])
def test_logits_reduce_small(nd, dtype, V, ld, excl):
    R = 37
    x = synth.logits(R, V, 4.0, 61, dtype=dtype, ld=ld)
    x[3, :V] = 0.5                         # all ties
    if V > 10:
        x[4, :V] = -1.0
        x[4, 7] = x[4, 9] = 2.0            # two-way tie
    ids, conf = nd.logits_reduce(x.cuda(), V, excl)
    rid, rconf = OD.logits_reduce(x.float().numpy()[:, :V], exclude_id=excl)
    assert np.array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(conf.cpu().numpy(), rconf, rtol=1e-4, atol=0)


def test_logits_reduce_batched_vocab(nd):
    c = synth.ATTN_BATCHED
    R = c["B"] * 32
    x = synth.logits(R, c["V"], c["logit_sigma"], c["seed"])
    ids, conf = nd.logits_reduce(x.cuda(), c["V"], c["V"] - 1)
    rid, rconf = OD.logits_reduce(x.float().numpy(), exclude_id=c["V"] - 1)
    assert np.array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(conf.cpu().numpy(), rconf, rtol=1e-4, atol=0)


# ---------------------------------------------------------------- unmask
@pytest.mark.parametrize("T", [32, 8, 1])
@pytest.mark.parametrize("ties,allm", [(False, False), (True, False), (True, True)])
def test_unmask(nd, T, ties, allm):
    B = 257
    conf, pred, mask = synth.unmask_inputs(B, T, 151936, 71 + T, ties=ties, all_masked=allm)
    for k in sorted({1, min(4, T), min(8, T), T}):
        blk = torch.full((B, T), 7, dtype=torch.int32)
        dr = torch.full((B, T), -1, dtype=torch.int32)
        m_d, b_d, d_d = mask.cuda(), blk.cuda(), dr.cuda()
        ch = torch.empty((B, k), dtype=torch.int32, device="cuda")
        nd.ndiff_unmask(conf.cuda(), pred.cuda(), B, T, k, m_d, b_d, d_d, ch)
        rm, rb, rd, rch = OD.unmask(conf.numpy(), pred.numpy(), mask.numpy().view(np.uint32),
                                    blk.numpy(), dr.numpy(), k)
        assert np.array_equal(m_d.cpu().numpy().view(np.uint32), rm)
        assert np.array_equal(b_d.cpu().numpy(), rb)
        assert np.array_equal(d_d.cpu().numpy(), rd)
        assert np.array_equal(ch.cpu().numpy(), rch)


@pytest.mark.parametrize("B", [256, 4096 + 77])
@pytest.mark.parametrize("ties,allm", [(False, False), (True, False), (True, True)])
def test_unmask_row_parallel_batches(nd, B, ties, allm):
    """Batches of 32-slot blocks from 256 sequences up take the four-lanes-a-
    sequence layout (k <= 8: winners extracted from per-lane sorted lists; k >
    8: ranks from pairwise key comparisons, keys passed by shuffle); a ragged
    last CTA and every k in {1, 4, 8, 32}, bit for bit."""
    T = 32
    conf, pred, mask = synth.unmask_inputs(B, T, 151936, 301 + B, ties=ties, all_masked=allm)
    for k in (1, 4, 8, 32):
        blk = torch.full((B, T), 7, dtype=torch.int32)
        dr = torch.full((B, T), -1, dtype=torch.int32)
        m_d, b_d, d_d = mask.cuda(), blk.cuda(), dr.cuda()
        ch = torch.empty((B, k), dtype=torch.int32, device="cuda")
        nd.ndiff_unmask(conf.cuda(), pred.cuda(), B, T, k, m_d, b_d, d_d, ch)
        rm, rb, rd, rch = OD.unmask(conf.numpy(), pred.numpy(), mask.numpy().view(np.uint32),
                                    blk.numpy(), dr.numpy(), k)
        assert np.array_equal(m_d.cpu().numpy().view(np.uint32), rm), k
        assert np.array_equal(b_d.cpu().numpy(), rb), k
        assert np.array_equal(d_d.cpu().numpy(), rd), k
        assert np.array_equal(ch.cpu().numpy(), rch), k


def test_unmask_signed_zero_and_infinite_confidence(nd):
    """-0 ties +0 (the lower slot wins), -inf ranks below every finite value
    and +inf above; both layouts (one warp per sequence below 256 sequences,
    four lanes per sequence from 256) against the oracle."""
    T = 32
    vals = np.array([0.0, -0.0, -np.inf, np.inf, 1e-30, -1e-30, 0.5, -0.5], dtype=np.float32)
    for B in (64, 512):
        rng = np.random.default_rng(B)
        conf = torch.from_numpy(vals[rng.integers(0, len(vals), size=(B, T))])
        pred = torch.from_numpy(rng.integers(0, 1000, size=(B, T)).astype(np.int32))
        mask = torch.from_numpy(rng.integers(0, 2**32, size=B, dtype=np.uint64)
                                .astype(np.uint32).view(np.int32))
        for k in (3, 32):
            blk = torch.zeros((B, T), dtype=torch.int32)
            dr = torch.full((B, T), -1, dtype=torch.int32)
            m_d, b_d, d_d = mask.cuda(), blk.cuda(), dr.cuda()
            ch = torch.empty((B, k), dtype=torch.int32, device="cuda")
            nd.ndiff_unmask(conf.cuda(), pred.cuda(), B, T, k, m_d, b_d, d_d, ch)
            rm, rb, rd, rch = OD.unmask(conf.numpy(), pred.numpy(), mask.numpy().view(np.uint32),
                                        blk.numpy(), dr.numpy(), k)
            assert np.array_equal(ch.cpu().numpy(), rch), (B, k)
            assert np.array_equal(m_d.cpu().numpy().view(np.uint32), rm), (B, k)
            assert np.array_equal(d_d.cpu().numpy(), rd), (B, k)
            assert np.array_equal(b_d.cpu().numpy(), rb), (B, k)


def test_unmask_and_verify_unaligned_rows_take_the_warp_layout(nd):
    """Row pointers that are not 16-byte aligned (a view offset by one
    element) fall back to one warp per sequence: same results."""
    B, T, k = 300, 32, 8
    conf, pred, mask = synth.unmask_inputs(B, T, 151936, 17)
    cbuf = torch.zeros(B * T + 1, device="cuda")
    pbuf = torch.zeros(B * T + 1, dtype=torch.int32, device="cuda")
    cbuf[1:] = conf.reshape(-1).cuda()
    pbuf[1:] = pred.reshape(-1).cuda()
    blk = torch.zeros((B, T), dtype=torch.int32)
    dr = torch.full((B, T), -1, dtype=torch.int32)
    m_d, b_d, d_d = mask.cuda(), blk.cuda(), dr.cuda()
    ch = torch.empty((B, k), dtype=torch.int32, device="cuda")
    nd.ndiff_unmask(cbuf[1:], pbuf[1:], B, T, k, m_d, b_d, d_d, ch)
    rm, rb, rd, rch = OD.unmask(conf.numpy(), pred.numpy(), mask.numpy().view(np.uint32),
                                blk.numpy(), dr.numpy(), k)
    assert np.array_equal(ch.cpu().numpy(), rch)
    assert np.array_equal(m_d.cpu().numpy().view(np.uint32), rm)
    assert np.array_equal(d_d.cpu().numpy(), rd) and np.array_equal(b_d.cpu().numpy(), rb)
    draft, target, _ = synth.draft_target(B, T, 151936, 18)
    dbuf = torch.zeros(B * T + 1, dtype=torch.int32, device="cuda")
    dbuf[1:] = draft.reshape(-1).cuda()
    kv = torch.arange(B, dtype=torch.int32)
    L = torch.empty(B, dtype=torch.int32, device="cuda")
    n = torch.empty(B, dtype=torch.int32, device="cuda")
    cm = torch.empty((B, T), dtype=torch.int32, device="cuda")
    kvd = kv.cuda()
    nd.ndiff_verify_accept(dbuf[1:], target.cuda(), B, T, L, cm, n, kvd)
    rL, rc, rn, rkv = OD.verify_accept(draft.numpy(), target.numpy(), kv.numpy())
    assert np.array_equal(L.cpu().numpy(), rL) and np.array_equal(n.cpu().numpy(), rn)
    assert np.array_equal(cm.cpu().numpy(), rc) and np.array_equal(kvd.cpu().numpy(), rkv)


@pytest.mark.parametrize("T,ties,allm", [(32, False, False), (32, True, False), (32, True, True),
                                         (7, True, False), (1, False, True)])
def test_unmask_threshold(nd, T, ties, allm):
    """Threshold rounds with revision against the oracle, bit for bit, with
    drafts that partly disagree with the predictions (so revision has work)
    and thresholds at and between the tie-heavy confidence values."""
    B = 257
    conf, pred, mask = synth.unmask_inputs(B, T, 151936, 91 + T, ties=ties, all_masked=allm)
    rng = np.random.default_rng(T)
    dr0 = np.where(rng.random((B, T)) < 0.5, pred.numpy(), rng.integers(0, 151936, size=(B, T)))
    dr0 = np.where((mask.numpy().view(np.uint32)[:, None] >> np.arange(T)) & 1, -1, dr0).astype(np.int32)
    for tau, taur in ((0.5, 2.0), (0.8125, 0.5), (0.0, 0.0), (1.0, 1.0), (1.5, 0.9375)):
        blk = torch.full((B, T), 7, dtype=torch.int32)
        dr = torch.from_numpy(dr0.copy())
        m_d, b_d, d_d = mask.cuda(), blk.cuda(), dr.cuda()
        nf = torch.empty(B, dtype=torch.int32, device="cuda")
        nr = torch.empty(B, dtype=torch.int32, device="cuda")
        nd.ndiff_unmask_threshold(conf.cuda(), pred.cuda(), B, T, tau, taur, m_d, b_d, d_d, nf, nr)
        rm, rb, rd, rnf, rnr = OD.unmask_threshold(conf.numpy(), pred.numpy(),
                                                   mask.numpy().view(np.uint32), blk.numpy(),
                                                   dr.numpy(), tau, taur)
        assert np.array_equal(m_d.cpu().numpy().view(np.uint32), rm), (tau, taur)
        assert np.array_equal(b_d.cpu().numpy(), rb), (tau, taur)
        assert np.array_equal(d_d.cpu().numpy(), rd), (tau, taur)
        assert np.array_equal(nf.cpu().numpy(), rnf) and np.array_equal(nr.cpu().numpy(), rnr)


def test_unmask_threshold_rejects_bad_arguments(nd):
    z = torch.zeros((1, 32), device="cuda")
    zi = torch.zeros((1, 32), dtype=torch.int32, device="cuda")
    m = torch.zeros(1, dtype=torch.int32, device="cuda")
    for tau, taur in ((-0.1, 2.0), (0.5, -1.0), (float("nan"), 2.0)):
        with pytest.raises(nd.NdiffError):
            nd.ndiff_unmask_threshold(z, zi, 1, 32, tau, taur, m, zi, zi)


# ---------------------------------------------------------------- verify/accept
@pytest.mark.parametrize("B,T", [(64, 32), (5, 1), (33, 7), (1000, 32), (1, 32), (31, 32),
                                 (4096 + 5, 32)])
def test_verify_accept(nd, B, T):
    draft, target, _ = synth.draft_target(B, T, 151936, 81 + T)
    kv = torch.arange(B, dtype=torch.int32) * 3
    L = torch.empty(B, dtype=torch.int32, device="cuda")
    n = torch.empty(B, dtype=torch.int32, device="cuda")
    cm = torch.empty((B, T), dtype=torch.int32, device="cuda")
    kvd = kv.cuda()
    nd.ndiff_verify_accept(draft.cuda(), target.cuda(), B, T, L, cm, n, kvd)
    rL, rc, rn, rkv = OD.verify_accept(draft.numpy(), target.numpy(), kv.numpy())
    assert np.array_equal(L.cpu().numpy(), rL)
    assert np.array_equal(n.cpu().numpy(), rn)
    assert np.array_equal(cm.cpu().numpy(), rc)
    assert np.array_equal(kvd.cpu().numpy(), rkv)


def test_unmask_and_verify_at_bench_batch_sampled_rows(nd):
    """The batch size the bandwidth figure is measured at (65536 sequences x
    32 slots): every row is independent, so 2048 sampled rows (first, last and
    random) are checked against the oracle bit for bit."""
    B, T, k = 65536, 32, 8
    conf, pred, mask = synth.unmask_inputs(B, T, 151936, 4001)
    draft, target, _ = synth.draft_target(B, T, 151936, 4002)
    blk = torch.zeros((B, T), dtype=torch.int32)
    dr = torch.zeros((B, T), dtype=torch.int32)
    m_d, b_d, d_d = mask.cuda(), blk.cuda(), dr.cuda()
    ch = torch.empty((B, k), dtype=torch.int32, device="cuda")
    nd.ndiff_unmask(conf.cuda(), pred.cuda(), B, T, k, m_d, b_d, d_d, ch)
    kv = torch.zeros(B, dtype=torch.int32)
    L = torch.empty(B, dtype=torch.int32, device="cuda")
    n = torch.empty(B, dtype=torch.int32, device="cuda")
    cm = torch.empty((B, T), dtype=torch.int32, device="cuda")
    kvd = kv.cuda()
    nd.ndiff_verify_accept(draft.cuda(), target.cuda(), B, T, L, cm, n, kvd)
    rows = np.unique(np.concatenate([[0, B - 1], np.random.default_rng(5).integers(0, B, 2046)]))
    rm, rb, rd, rch = OD.unmask(conf.numpy()[rows], pred.numpy()[rows],
                                mask.numpy().view(np.uint32)[rows], blk.numpy()[rows],
                                dr.numpy()[rows], k)
    assert np.array_equal(m_d.cpu().numpy().view(np.uint32)[rows], rm)
    assert np.array_equal(b_d.cpu().numpy()[rows], rb)
    assert np.array_equal(d_d.cpu().numpy()[rows], rd)
    assert np.array_equal(ch.cpu().numpy()[rows], rch)
    rL, rc, rn, rkv = OD.verify_accept(draft.numpy()[rows], target.numpy()[rows], kv.numpy()[rows])
    assert np.array_equal(L.cpu().numpy()[rows], rL)
    assert np.array_equal(n.cpu().numpy()[rows], rn)
    assert np.array_equal(cm.cpu().numpy()[rows], rc)
    assert np.array_equal(kvd.cpu().numpy()[rows], rkv)
