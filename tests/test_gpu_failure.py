"""Failure detection on the GPU without a fault: a kernel's bounded wait on a
barrier that nothing arrives on expires, the kernel records the expiry in the
device status word and returns, the host reads NDIFF_ERR_TIMEOUT, and the
context keeps working (a real computation right after still matches the
oracle). Host-side argument errors are covered without a GPU in test_abi."""
import time

import numpy as np
import pytest
import torch

from oracle import decode as OD
from self_speculative_lm_block_b300 import synth

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_context_survives(cuda_ok):
    from self_speculative_lm_block_b300 import ndiff as nd
    nd.ndiff_check()                                  # start from a clear status word
    t0 = time.perf_counter()
    nd.ndiff_selftest_timeout(20000)                  # 20 ms limit
    with pytest.raises(nd.NdiffError) as e:
        nd.ndiff_check()
    assert e.value.status == nd.NDIFF_ERR_TIMEOUT
    assert time.perf_counter() - t0 >= 0.015
    nd.ndiff_check()                                  # the word was cleared
    # the context is still usable
    x = synth.logits(8, 1000, 4.0, 3)
    ids, conf = nd.logits_reduce(x.cuda(), 1000, 999)
    rid, rconf = OD.logits_reduce(x.float().numpy(), exclude_id=999)
    assert np.array_equal(ids.cpu().numpy(), rid)
    nd.ndiff_check()


def test_selftest_rejects_bad_limits(cuda_ok):
    from self_speculative_lm_block_b300 import ndiff as nd
    for bad in (0, -1, 2000001):
        with pytest.raises(nd.NdiffError) as e:
            nd.ndiff_selftest_timeout(bad)
        assert e.value.status == nd.NDIFF_ERR_INVALID_ARG


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_out_of_range_kv_len_is_reported(cuda_ok, dtype):
    """A kv_len outside [0, Lmax - T] is an error only the device can see: the
    kernels keep every access inside the cache, record the error in the status
    word, and the next check returns NDIFF_ERR_INVALID_ARG; the word is then
    clear and a valid call right after matches the oracle."""
    from oracle import attention as OA
    from self_speculative_lm_block_b300 import ndiff as nd
    nd.ndiff_check()
    if dtype == "bf16":
        B, T, Hq, Hkv, D, Lmax, tdt = 2, 32, 32, 8, 128, 400, torch.bfloat16
    else:
        B, T, Hq, Hkv, D, Lmax, tdt = 2, 32, 4, 4, 32, 400, torch.float32
    inp = synth.attn_inputs(B, T, Hq, Hkv, D, [100, 200], Lmax, 41, dtype=tdt)
    q, k, v = inp.q.cuda(), inp.k_cache.cuda(), inp.v_cache.cuda()
    for bad in ([Lmax - T + 1, 10], [5, -3], [Lmax, Lmax]):
        kv = torch.tensor(bad, dtype=torch.int32, device="cuda")
        nd.block_attn(q, k, v, kv, nd.NDIFF_CAUSAL, inp.scale)
        with pytest.raises(nd.NdiffError) as e:
            nd.ndiff_check()
        assert e.value.status == nd.NDIFF_ERR_INVALID_ARG, bad
        nd.ndiff_check()                              # cleared
    out = nd.block_attn(q, k, v, inp.kv_len.cuda(), nd.NDIFF_CAUSAL, inp.scale)
    nd.ndiff_check()
    ref = OA.block_attn(inp.q.float().numpy(), inp.k_cache.float().numpy(),
                        inp.v_cache.float().numpy(), inp.kv_len.numpy(), OA.CAUSAL, inp.scale)
    err = np.abs(out.float().cpu().numpy() - ref)
    tol = 1e-2 + 1e-2 * np.abs(ref) if dtype == "bf16" else 1e-5 + 1e-5 * np.abs(ref)
    assert (err <= tol).all()
