"""The allocation-free block attention entry point, checked against the
regular one.

ndiff_block_attn_noalloc exists for callers that cannot allocate device memory
(plugin interfaces that receive only inputs and outputs, or processes whose
memory manager owns the whole device). It takes its split-KV scratch from an
array built into the library instead of a caller workspace. This file is named
so that pytest collects it last."""
import numpy as np
import pytest
import torch

from self_speculative_lm_block_b300 import synth

pytestmark = pytest.mark.gpu


def _regular(nd, inp, mode):
    return nd.block_attn(inp.q.cuda(), inp.k_cache.cuda(), inp.v_cache.cuda(), inp.kv_len.cuda(),
                         mode, inp.scale)


def _noalloc(nd, inp, mode):
    B, T, Hq, D = inp.q.shape
    Hkv, Lmax = inp.k_cache.shape[1], inp.k_cache.shape[2]
    out = torch.empty(inp.q.shape, dtype=inp.q.dtype, device="cuda")
    nd.ndiff_block_attn_noalloc(nd.NDIFF_BF16, inp.q.cuda(), inp.k_cache.cuda(), inp.v_cache.cuda(),
                                inp.kv_len.cuda(), B, T, Hq, Hkv, D, Lmax, mode, inp.scale, out)
    return out


def test_noalloc_matches_regular_entry_point_twice(cuda_ok):
    from self_speculative_lm_block_b300 import ndiff as nd
    # two different calls in a row: the second must not see the first's scratch
    cases = [(synth.attn_inputs(2, 32, 32, 8, 128, [700, 300], 800, 91, fill_tail=float("nan")), 1),
             (synth.attn_inputs(3, 5, 32, 8, 128, [520, 4, 777], 800, 92, fill_tail=float("nan")), 0)]
    for inp, mode in cases:
        B, T, Hq, D = inp.q.shape
        # the shape really uses the scratch (several KV splits)
        assert 0 < nd.ndiff_block_attn_workspace_size(nd.NDIFF_BF16, B, T, Hq, 8, D, 800) \
            <= nd.NDIFF_NOALLOC_SCRATCH_BYTES
        got = _noalloc(nd, inp, mode).float().cpu().numpy()
        ref = _regular(nd, inp, mode).float().cpu().numpy()
        nd.ndiff_check()
        assert np.isfinite(got).all()
        assert (np.abs(got - ref) <= 1e-2 + 1e-2 * np.abs(ref)).all()


def test_noalloc_rejects_shapes_beyond_its_scratch(cuda_ok):
    from self_speculative_lm_block_b300 import ndiff as nd
    B, T, Hq, Hkv, D, Lmax = 64, 32, 32, 8, 128, 32800
    assert nd.ndiff_block_attn_workspace_size(nd.NDIFF_BF16, B, T, Hq, Hkv, D, Lmax) > \
        nd.NDIFF_NOALLOC_SCRATCH_BYTES
    with pytest.raises(nd.NdiffError) as e:
        nd.ndiff_block_attn_noalloc(nd.NDIFF_BF16, 16, 16, 16, 16, B, T, Hq, Hkv, D, Lmax, 0, 0.1, 16)
    assert e.value.status == nd.NDIFF_ERR_WORKSPACE
