"""The allocation-free block attention entry point, checked against the
regular one.

ndiff_block_attn_noalloc exists for callers that cannot allocate device memory
(plugin interfaces that receive only inputs and outputs, or processes whose
memory manager owns the whole device). It takes its split-KV scratch from an
array built into the library instead of a caller workspace. It runs the same
kernels with the same KV split as ndiff_block_attn, so its output must equal
that entry point's bit for bit; a stale partial left in the shared array by an
earlier call would break that. This file is named so that pytest collects it
last."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

Hq, Hkv, D, T = 32, 8, 128, 32


def _inputs(B, lengths, Lmax, seed, t=T):
    """Seeded N(0,1) bf16 q/k/v drawn on the device (no oracle is involved, so
    full-size caches need not pass through the host); cache rows past each
    sequence's block hold NaN, which must never be read."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randn((B, t, Hq, D), generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn((B, Hkv, Lmax, D), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((B, Hkv, Lmax, D), generator=g, device="cuda").to(torch.bfloat16)
    for b, P in enumerate(lengths):
        k[b, :, P + t:] = float("nan")
        v[b, :, P + t:] = float("nan")
    kv = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    return q, k, v, kv


def _regular(nd, q, k, v, kv, mode):
    B, t = q.shape[0], q.shape[1]
    Lmax = k.shape[2]
    out = torch.empty_like(q)
    need = nd.ndiff_block_attn_workspace_size(nd.NDIFF_BF16, B, t, Hq, Hkv, D, Lmax)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    nd.ndiff_block_attn(nd.NDIFF_BF16, q, k, v, kv, B, t, Hq, Hkv, D, Lmax, mode, D ** -0.5, out,
                        ws, need)
    return out


def _noalloc(nd, q, k, v, kv, mode, out=None):
    B, t = q.shape[0], q.shape[1]
    Lmax = k.shape[2]
    out = torch.empty_like(q) if out is None else out
    nd.ndiff_block_attn_noalloc(nd.NDIFF_BF16, q, k, v, kv, B, t, Hq, Hkv, D, Lmax, mode, D ** -0.5,
                                out)
    return out


def test_noalloc_equals_regular_entry_point_call_after_call(cuda_ok):
    """A first call that writes partials over 95% of the built-in scratch, then
    smaller calls (one sequence with several KV splits, where the partials
    start at offset 0; a ragged batch; a short block) that each must equal the
    regular entry point exactly."""
    from self_speculative_lm_block_b300 import ndiff as nd
    cap = nd.NDIFF_NOALLOC_SCRATCH_BYTES
    cases = [
        (10, [38880] * 10, 38912, 1, T),       # ~16.0 MB of partials: nearly the whole array
        (1, [4096], 4128, 0, T),               # batch 1: no launch-order table, several splits
        (3, [700, 300, 5], 800, 1, T),         # ragged batch
        (2, [1500, 2900], 3000, 0, 5),         # a short block, BIDIR
        (1, [4096], 4128, 1, T),               # batch 1 again, after other shapes
    ]
    for i, (B, lengths, Lmax, mode, t) in enumerate(cases):
        need = nd.ndiff_block_attn_workspace_size(nd.NDIFF_BF16, B, t, Hq, Hkv, D, Lmax)
        assert 0 < need <= cap, (i, need)
        if i == 0:
            assert need >= 0.9 * cap
        q, k, v, kv = _inputs(B, lengths, Lmax, 500 + i, t)
        got = _noalloc(nd, q, k, v, kv, mode)
        ref = _regular(nd, q, k, v, kv, mode)
        nd.ndiff_check()
        assert torch.isfinite(got.float()).all()
        assert torch.equal(got, ref), (i, (got.float() - ref.float()).abs().max().item())
        del q, k, v, kv, got, ref
        torch.cuda.empty_cache()


def test_noalloc_allocates_no_device_memory(cuda_ok):
    """After one warm-up call (kernels loaded, scratch address looked up), a
    call on a new shape changes neither torch's allocation count nor the
    device's free memory."""
    from self_speculative_lm_block_b300 import ndiff as nd
    q0, k0, v0, kv0 = _inputs(2, [900, 1700], 1800, 601)
    _noalloc(nd, q0, k0, v0, kv0, 1)
    q, k, v, kv = _inputs(3, [2000, 64, 1333], 2100, 602)
    out = torch.empty_like(q)
    torch.cuda.synchronize()
    alloc0 = torch.cuda.memory_allocated()
    free0 = torch.cuda.mem_get_info()[0]
    _noalloc(nd, q, k, v, kv, 0, out)
    _noalloc(nd, q, k, v, kv, 1, out)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.mem_get_info()[0] == free0
    nd.ndiff_check()
    assert torch.equal(out, _regular(nd, q, k, v, kv, 1))


def test_noalloc_rejects_shapes_beyond_its_scratch(cuda_ok):
    from self_speculative_lm_block_b300 import ndiff as nd
    B, Lmax = 64, 32800
    assert nd.ndiff_block_attn_workspace_size(nd.NDIFF_BF16, B, T, Hq, Hkv, D, Lmax) > \
        nd.NDIFF_NOALLOC_SCRATCH_BYTES
    with pytest.raises(nd.NdiffError) as e:
        nd.ndiff_block_attn_noalloc(nd.NDIFF_BF16, 16, 16, 16, 16, B, T, Hq, Hkv, D, Lmax, 0, 0.1, 16)
    assert e.value.status == nd.NDIFF_ERR_WORKSPACE
