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
