"""CPU checks of the C-ABI library: it builds, loads without a GPU, exports every
entry point that include/ndiff.h declares, and rejects bad arguments on the
host before touching a device."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def nd():
    from self_speculative_lm_block_b300 import build
    build.build()
    from self_speculative_lm_block_b300 import ndiff
    return ndiff


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"NDIFF_API\s+[\w\s\*]+?\b(ndiff_\w+)\s*\(", txt))
    return names


def test_every_declared_symbol_is_exported(nd):
    import ctypes
    lib = ctypes.CDLL(nd.LIB_PATH)
    declared = _declared()
    assert len(declared) >= 17
    for name in sorted(declared):
        assert hasattr(lib, name), name
    assert declared <= set(nd.exported_names())


def test_status_strings(nd):
    assert nd.ndiff_status_string(0) == "NDIFF_OK"
    assert nd.ndiff_status_string(6) == "NDIFF_ERR_TIMEOUT"


def test_host_side_validation_without_gpu(nd):
    # every rejection below happens before any CUDA call
    with pytest.raises(nd.NdiffError) as e:
        nd.ndiff_unmask(1, 1, 4, 33, 1, 1, 1, 1, 1, stream=0)
    assert e.value.status == nd.NDIFF_ERR_INVALID_ARG
    with pytest.raises(nd.NdiffError) as e:
        nd.ndiff_verify_accept(1, 1, 4, 0, 1, 1, 1, None, stream=0)
    assert e.value.status == nd.NDIFF_ERR_INVALID_ARG
    with pytest.raises(nd.NdiffError) as e:
        nd.ndiff_logits_reduce(nd.NDIFF_BF16, 16, 4, 100, 50, -1, 16, 16, stream=0)
    assert e.value.status == nd.NDIFF_ERR_INVALID_ARG
    with pytest.raises(nd.NdiffError) as e:
        nd.ndiff_block_attn(nd.NDIFF_BF16, 16, 16, 16, 16, 1, 32, 32, 8, 64, 100, 0, 0.1, 16,
                            stream=0)
    assert e.value.status == nd.NDIFF_ERR_UNSUPPORTED
    with pytest.raises(nd.NdiffError) as e:
        nd.ndiff_block_attn(nd.NDIFF_BF16, 16, 16, 16, 16, 1, 64, 32, 8, 128, 100, 0, 0.1, 16,
                            stream=0)
    assert e.value.status == nd.NDIFF_ERR_UNSUPPORTED  # G*T = 256 > 128
    # empty batches are no-ops
    nd.ndiff_unmask(None, None, 0, 32, 1, None, None, None, None, stream=0)
    nd.ndiff_verify_accept(None, None, 0, 32, None, None, None, None, stream=0)
    nd.ndiff_logits_reduce(nd.NDIFF_F32, None, 0, 10, 10, -1, None, None, stream=0)


def test_host_side_validation_of_the_later_entry_points(nd):
    """Threshold unmask, fused LM head, plain projection and the model calls
    reject bad arguments on the host, before any device work."""
    for tau, taur in ((-1.0, 2.0), (0.5, -0.5), (float("nan"), 2.0)):
        with pytest.raises(nd.NdiffError) as e:
            nd.ndiff_unmask_threshold(16, 16, 1, 32, tau, taur, 16, 16, 16, stream=0)
        assert e.value.status == nd.NDIFF_ERR_INVALID_ARG
    with pytest.raises(nd.NdiffError) as e:
        nd.ndiff_unmask_threshold(16, 16, 1, 33, 0.5, 2.0, 16, 16, 16, stream=0)   # T > 32
    assert e.value.status == nd.NDIFF_ERR_INVALID_ARG
    nd.ndiff_unmask_threshold(None, None, 0, 32, 0.5, 2.0, None, None, None, stream=0)  # empty batch
    for M, N, K, ex in ((0, 128, 64, -1), (4, 128, 96, -1), (4, 128, 64, 128), (4, 128, 64, -2)):
        with pytest.raises(nd.NdiffError) as e:
            nd.ndiff_lm_head_argmax(16, 16, M, N, K, ex, 16, 16, 16, 1 << 20, stream=0)
        assert e.value.status == nd.NDIFF_ERR_INVALID_ARG
    with pytest.raises(nd.NdiffError) as e:
        nd.ndiff_gemm_bf16(16, 16, 4, 128, 64, 16, 100, 16, 1 << 20, stream=0)      # ldy < N
    assert e.value.status == nd.NDIFF_ERR_INVALID_ARG
    with pytest.raises(nd.NdiffError):
        nd._call("ndiff_decode_step_ex", None, None, None, None, None, nd._stream(0))
    with pytest.raises(nd.NdiffError):
        nd._call("ndiff_prefill_batch", None, None, None, nd._stream(0))
    with pytest.raises(nd.NdiffError):
        nd._call("ndiff_decode_step_batch", None, None, None, None, None, nd._stream(0))


def test_workspace_sizes(nd):
    # one sequence, one split: no scratch
    assert nd.ndiff_block_attn_split_workspace_size(nd.NDIFF_BF16, 1, 32, 32, 8, 128, 512, 512) == 0
    # one sequence, four splits: the partial results (fp32 O rows + (m, l) per row)
    w = nd.ndiff_block_attn_split_workspace_size(nd.NDIFF_BF16, 1, 32, 32, 8, 128, 512, 128)
    assert w == 1 * 8 * 4 * 128 * (128 * 4 + 8)
    # a batch adds its launch order (one int per (sequence, split), 256-byte granules)
    assert nd.ndiff_block_attn_split_workspace_size(nd.NDIFF_BF16, 2, 32, 32, 8, 128, 512, 512) == 256
    w = nd.ndiff_block_attn_split_workspace_size(nd.NDIFF_BF16, 2, 32, 32, 8, 128, 512, 128)
    assert w == 2 * 8 * 4 * 128 * (128 * 4 + 8) + 256
    assert nd.ndiff_block_attn_workspace_size(nd.NDIFF_F32, 2, 32, 4, 4, 32, 512) == 0


def test_noalloc_reports_argument_errors_before_the_scratch_limit(nd):
    """A shape too large for the built-in scratch with a bad argument reports
    the argument error (as ndiff_block_attn would), not NDIFF_ERR_WORKSPACE;
    with valid arguments it reports NDIFF_ERR_WORKSPACE. All on the host."""
    B, T, Hq, Hkv, D, Lmax = 64, 32, 32, 8, 128, 32800
    assert nd.ndiff_block_attn_workspace_size(nd.NDIFF_BF16, B, T, Hq, Hkv, D, Lmax) > \
        nd.NDIFF_NOALLOC_SCRATCH_BYTES
    bad = [
        (dict(Hq=30), nd.NDIFF_ERR_INVALID_ARG),          # Hq % Hkv != 0
        (dict(mode=7), nd.NDIFF_ERR_INVALID_ARG),         # bad mask mode
        (dict(dt=5), nd.NDIFF_ERR_INVALID_ARG),           # bad dtype
        (dict(q=17), nd.NDIFF_ERR_INVALID_ARG),           # misaligned bf16 pointer
        (dict(T=64), nd.NDIFF_ERR_UNSUPPORTED),           # G * T = 256 > 128
    ]
    for change, want in bad + [({}, nd.NDIFF_ERR_WORKSPACE)]:
        a = dict(dt=nd.NDIFF_BF16, q=16, B=B, T=T, Hq=Hq, mode=0)
        a.update(change)
        with pytest.raises(nd.NdiffError) as e:
            nd.ndiff_block_attn_noalloc(a["dt"], a["q"], 16, 16, 16, a["B"], a["T"], a["Hq"], Hkv, D, Lmax,
                                        a["mode"], 0.1, 16, stream=0)
        assert e.value.status == want, (change, e.value.status)
