"""ctypes binding of libndiff (include/ndiff.h): the same entry points under the
same names, argument marshalling only. Pointer arguments take torch tensors
(their data_ptr), ints or None; the stream defaults to torch's current stream.

Every compute step runs in libndiff's CUDA kernels. There is no fallback: if
the library is missing or fails to load, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libndiff.so")

NDIFF_OK, NDIFF_ERR_INVALID_ARG, NDIFF_ERR_UNSUPPORTED = 0, 1, 2
NDIFF_ERR_CUDA, NDIFF_ERR_OOM, NDIFF_ERR_WORKSPACE, NDIFF_ERR_TIMEOUT = 3, 4, 5, 6
NDIFF_BF16, NDIFF_F32 = 0, 1
NDIFF_BIDIR, NDIFF_CAUSAL = 0, 1
NDIFF_MODE_AR, NDIFF_MODE_DIFF, NDIFF_MODE_SELFSPEC, NDIFF_MODE_SELFSPEC_FUSED = 0, 1, 2, 3
NDIFF_MODE_SELFSPEC_QUAD = 4
NDIFF_NOALLOC_SCRATCH_BYTES = 16 << 20


class NdiffError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: status {status}: {msg}")
        self.status = status


class ModelConfig(ctypes.Structure):
    _fields_ = [("layers", ctypes.c_int), ("d_model", ctypes.c_int), ("n_heads", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("vocab", ctypes.c_int), ("dtype", ctypes.c_int), ("rope_base", ctypes.c_float),
                ("eps", ctypes.c_float), ("max_seq", ctypes.c_int), ("batch", ctypes.c_int)]


class Stats(ctypes.Structure):
    _fields_ = [("forwards", ctypes.c_int64), ("tokens", ctypes.c_int64),
                ("last_accept_len", ctypes.c_int32), ("last_n_commit", ctypes.c_int32),
                ("accept_hist", ctypes.c_int64 * 33), ("revisions", ctypes.c_int64),
                ("last_rounds", ctypes.c_int32), ("reserved", ctypes.c_int32)]


NDIFF_SAMPLER_TOPK = 0
NDIFF_SAMPLER_THRESHOLD = 1


class DecodeOpts(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int), ("sampler", ctypes.c_int), ("steps", ctypes.c_int),
                ("tau", ctypes.c_float), ("tau_revise", ctypes.c_float), ("n_cand", ctypes.c_int),
                ("cand", ctypes.c_int * 2)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_F = ctypes.c_float
_I64 = ctypes.c_int64

_SIGS = {
    "ndiff_last_error": (ctypes.c_char_p, []),
    "ndiff_status_string": (ctypes.c_char_p, [_I]),
    "ndiff_check": (_I, [_P]),
    "ndiff_selftest_timeout": (_I, [_I, _P]),
    "ndiff_block_attn": (_I, [_I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _SZ, _P]),
    "ndiff_block_attn_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "ndiff_block_attn_split": (_I, [_I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _P,
                                    _SZ, _P]),
    "ndiff_block_attn_split_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I, _I]),
    "ndiff_block_attn_noalloc": (_I, [_I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P]),
    "ndiff_logits_reduce": (_I, [_I, _P, _I, _I, _I64, _I, _P, _P, _P]),
    "ndiff_gemm_bf16_workspace_size": (_SZ, [_I, _I, _I]),
    "ndiff_gemm_bf16": (_I, [_P, _P, _I, _I, _I, _P, _I64, _P, _SZ, _P]),
    "ndiff_lm_head_argmax_workspace_size": (_SZ, [_I, _I, _I]),
    "ndiff_lm_head_argmax": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _SZ, _P]),
    "ndiff_unmask": (_I, [_P, _P, _I, _I, _I, _P, _P, _P, _P, _P]),
    "ndiff_unmask_threshold": (_I, [_P, _P, _I, _I, _F, _F, _P, _P, _P, _P, _P, _P]),
    "ndiff_decode_step_ex": (_I, [_P, _P, _P, _P, _P, _P]),
    "ndiff_prefill_batch": (_I, [_P, _P, _P, _P]),
    "ndiff_decode_step_batch": (_I, [_P, _P, _P, _P, _P, _P]),
    "ndiff_model_state_batch": (_I, [_P, _P, _P]),
    "ndiff_verify_accept": (_I, [_P, _P, _I, _I, _P, _P, _P, _P, _P]),
    "ndiff_model_create": (_I, [ctypes.POINTER(ModelConfig), ctypes.c_uint64, ctypes.POINTER(_P)]),
    "ndiff_model_destroy": (_I, [_P]),
    "ndiff_prefill": (_I, [_P, _P, _I, _P]),
    "ndiff_decode_step": (_I, [_P, _I, _I, _P, ctypes.POINTER(_I), ctypes.POINTER(Stats), _P]),
    "ndiff_model_forward": (_I, [_P, _P, _I, _I, _P, _P]),
    "ndiff_model_state": (_I, [_P, ctypes.POINTER(_I), ctypes.POINTER(ctypes.c_int32)]),
    "ndiff_model_read_weight": (_I, [_P, _I, _I64, _I64, _P]),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libndiff.so not built at {LIB_PATH}; run "
                          "`python -m self_speculative_lm_block_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGS.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib = _load()


def exported_names():
    return list(_SIGS)


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return x.data_ptr()
    return int(x)


def _stream(s):
    if s is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(s, torch.cuda.Stream):
        return s.cuda_stream
    return int(s)


def _call(name, *args):
    st = getattr(_lib, name)(*args)
    if st != NDIFF_OK:
        raise NdiffError(name, st, _lib.ndiff_last_error().decode())
    return st


def ndiff_last_error() -> str:
    return _lib.ndiff_last_error().decode()


def ndiff_status_string(s: int) -> str:
    return _lib.ndiff_status_string(s).decode()


def ndiff_check(stream=None):
    return _call("ndiff_check", _stream(stream))


def ndiff_selftest_timeout(limit_us: int, stream=None):
    return _call("ndiff_selftest_timeout", limit_us, _stream(stream))


def ndiff_block_attn(dt, q, k_cache, v_cache, kv_len, B, T, Hq, Hkv, D, Lmax, mode, scale, out,
                     ws=None, ws_bytes=0, stream=None):
    return _call("ndiff_block_attn", dt, _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_len), B, T,
                 Hq, Hkv, D, Lmax, mode, scale, _ptr(out), _ptr(ws), ws_bytes, _stream(stream))


def ndiff_block_attn_workspace_size(dt, B, T, Hq, Hkv, D, Lmax) -> int:
    return _lib.ndiff_block_attn_workspace_size(dt, B, T, Hq, Hkv, D, Lmax)


def ndiff_block_attn_split(dt, q, k_cache, v_cache, kv_len, B, T, Hq, Hkv, D, Lmax, mode, scale,
                           split_keys, out, ws=None, ws_bytes=0, stream=None):
    return _call("ndiff_block_attn_split", dt, _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_len),
                 B, T, Hq, Hkv, D, Lmax, mode, scale, split_keys, _ptr(out), _ptr(ws), ws_bytes,
                 _stream(stream))


def ndiff_block_attn_split_workspace_size(dt, B, T, Hq, Hkv, D, Lmax, split_keys) -> int:
    return _lib.ndiff_block_attn_split_workspace_size(dt, B, T, Hq, Hkv, D, Lmax, split_keys)


def ndiff_block_attn_noalloc(dt, q, k_cache, v_cache, kv_len, B, T, Hq, Hkv, D, Lmax, mode, scale,
                             out, stream=None):
    return _call("ndiff_block_attn_noalloc", dt, _ptr(q), _ptr(k_cache), _ptr(v_cache),
                 _ptr(kv_len), B, T, Hq, Hkv, D, Lmax, mode, scale, _ptr(out), _stream(stream))


def ndiff_logits_reduce(dt, logits, R, V, ld, exclude_id, argmax, conf, stream=None):
    return _call("ndiff_logits_reduce", dt, _ptr(logits), R, V, ld, exclude_id, _ptr(argmax),
                 _ptr(conf), _stream(stream))


def ndiff_gemm_bf16_workspace_size(M, N, K) -> int:
    return _lib.ndiff_gemm_bf16_workspace_size(M, N, K)


def ndiff_gemm_bf16(x, w, M, N, K, y, ldy, ws, ws_bytes, stream=None):
    return _call("ndiff_gemm_bf16", _ptr(x), _ptr(w), M, N, K, _ptr(y), ldy, _ptr(ws), ws_bytes,
                 _stream(stream))


def ndiff_lm_head_argmax_workspace_size(M, N, K) -> int:
    return _lib.ndiff_lm_head_argmax_workspace_size(M, N, K)


def ndiff_lm_head_argmax(x, w, M, N, K, exclude_id, argmax, conf, ws, ws_bytes, stream=None):
    return _call("ndiff_lm_head_argmax", _ptr(x), _ptr(w), M, N, K, exclude_id, _ptr(argmax),
                 _ptr(conf), _ptr(ws), ws_bytes, _stream(stream))


def ndiff_unmask_threshold(conf, pred, B, T, tau, tau_revise, mask_bits, block_in, draft,
                           n_fixed=None, n_revised=None, stream=None):
    return _call("ndiff_unmask_threshold", _ptr(conf), _ptr(pred), B, T, tau, tau_revise,
                 _ptr(mask_bits), _ptr(block_in), _ptr(draft), _ptr(n_fixed), _ptr(n_revised),
                 _stream(stream))


def ndiff_unmask(conf, pred, B, T, k, mask_bits, block_in, draft, chosen, stream=None):
    return _call("ndiff_unmask", _ptr(conf), _ptr(pred), B, T, k, _ptr(mask_bits), _ptr(block_in),
                 _ptr(draft), _ptr(chosen), _stream(stream))


def ndiff_verify_accept(draft, target, B, T, accept_len, commit, n_commit, kv_len=None, stream=None):
    return _call("ndiff_verify_accept", _ptr(draft), _ptr(target), B, T, _ptr(accept_len),
                 _ptr(commit), _ptr(n_commit), _ptr(kv_len), _stream(stream))


def ndiff_model_create(cfg: ModelConfig, seed: int) -> int:
    h = _P()
    _call("ndiff_model_create", ctypes.byref(cfg), seed, ctypes.byref(h))
    return h.value


def ndiff_model_destroy(m: int):
    return _call("ndiff_model_destroy", m)


def ndiff_prefill(m: int, prompt_host, n: int, stream=None):
    return _call("ndiff_prefill", m, _ptr(prompt_host), n, _stream(stream))


def ndiff_decode_step(m: int, mode: int, steps: int, out_tokens_host, stats: Stats | None = None,
                      stream=None) -> int:
    n = _I(0)
    _call("ndiff_decode_step", m, mode, steps, _ptr(out_tokens_host), ctypes.byref(n),
          ctypes.byref(stats) if stats is not None else None, _stream(stream))
    return n.value


def ndiff_decode_step_ex(m: int, opts: DecodeOpts, out_tokens_host, stats: Stats | None = None,
                         stream=None) -> int:
    n = _I(0)
    _call("ndiff_decode_step_ex", m, ctypes.byref(opts), _ptr(out_tokens_host), ctypes.byref(n),
          ctypes.byref(stats) if stats is not None else None, _stream(stream))
    return n.value


def ndiff_model_forward(m: int, ids_host, T: int, mode: int, logits_host, stream=None):
    return _call("ndiff_model_forward", m, _ptr(ids_host), T, mode, _ptr(logits_host), _stream(stream))


def ndiff_model_state(m: int):
    kv = _I(0)
    last = ctypes.c_int32(0)
    _call("ndiff_model_state", m, ctypes.byref(kv), ctypes.byref(last))
    return kv.value, last.value


def ndiff_model_read_weight(m: int, tensor_id: int, offset: int, count: int, host_out):
    return _call("ndiff_model_read_weight", m, tensor_id, offset, count, _ptr(host_out))


# --------------------------------------------------------------------------
# Convenience wrappers (shape bookkeeping and scratch allocation only)
# --------------------------------------------------------------------------
def block_attn(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, kv_len: torch.Tensor,
               mode: int, scale: float, split_keys: int = 0, out: torch.Tensor | None = None,
               stream=None) -> torch.Tensor:
    B, T, Hq, D = q.shape
    Hkv, Lmax = k_cache.shape[1], k_cache.shape[2]
    dt = NDIFF_BF16 if q.dtype == torch.bfloat16 else NDIFF_F32
    out = torch.empty_like(q) if out is None else out
    need = ndiff_block_attn_split_workspace_size(dt, B, T, Hq, Hkv, D, Lmax, split_keys)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device) if need else None
    ndiff_block_attn_split(dt, q, k_cache, v_cache, kv_len, B, T, Hq, Hkv, D, Lmax, mode, scale,
                           split_keys, out, ws, need, stream)
    return out


def logits_reduce(logits: torch.Tensor, V: int | None = None, exclude_id: int = -1, stream=None):
    R, ld = logits.shape
    V = ld if V is None else V
    dt = NDIFF_BF16 if logits.dtype == torch.bfloat16 else NDIFF_F32
    ids = torch.empty(R, dtype=torch.int32, device=logits.device)
    conf = torch.empty(R, dtype=torch.float32, device=logits.device)
    ndiff_logits_reduce(dt, logits, R, V, ld, exclude_id, ids, conf, stream)
    return ids, conf


def gemm_bf16(x: torch.Tensor, w: torch.Tensor, stream=None) -> torch.Tensor:
    """y = x @ w.T in fp32 for bf16 x [M<=32][K] and w [N][K] (device tensors)."""
    M, K = x.shape
    N = w.shape[0]
    y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    need = ndiff_gemm_bf16_workspace_size(M, N, K)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    ndiff_gemm_bf16(x, w, M, N, K, y, N, ws, need, stream)
    return y


def lm_head_argmax(x: torch.Tensor, w: torch.Tensor, exclude_id: int = -1, stream=None):
    """(argmax, conf) of the rows of x @ w.T without storing the logits; bf16
    x [M<=32][K] and w [N][K] (device tensors)."""
    M, K = x.shape
    N = w.shape[0]
    ids = torch.empty(M, dtype=torch.int32, device=x.device)
    conf = torch.empty(M, dtype=torch.float32, device=x.device)
    need = ndiff_lm_head_argmax_workspace_size(M, N, K)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    ndiff_lm_head_argmax(x, w, M, N, K, exclude_id, ids, conf, ws, need, stream)
    return ids, conf


class Model:
    """Owner of an ndiff_model handle (thin wrapper over the C ABI)."""

    def __init__(self, layers, d_model, n_heads, n_kv_heads, head_dim, ffn, vocab, dtype="f32",
                 max_seq=4096, seed=0, rope_base=10000.0, eps=1e-6, batch=1):
        cfg = ModelConfig(layers, d_model, n_heads, n_kv_heads, head_dim, ffn, vocab,
                          NDIFF_BF16 if dtype == "bf16" else NDIFF_F32, rope_base, eps, max_seq,
                          batch)
        self.cfg = cfg
        self.vocab = vocab
        self.batch = batch
        self.handle = ndiff_model_create(cfg, seed)
        self.stats = Stats()

    def close(self):
        if self.handle:
            ndiff_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def prefill(self, prompt):
        import numpy as np
        arr = np.ascontiguousarray(np.asarray(prompt, dtype=np.int32))
        ndiff_prefill(self.handle, arr.ctypes.data, int(arr.shape[0]))

    def step(self, mode: int, steps: int = 1, tau: float | None = None, tau_revise: float = 2.0,
             cands=None):
        """One decode cycle; with `tau` the draft uses the threshold sampler;
        `cands` (one or two lengths in [0, 32)) are the candidate acceptance
        lengths of NDIFF_MODE_SELFSPEC_QUAD."""
        buf = (ctypes.c_int32 * 32)()
        if tau is None and cands is None:
            n = ndiff_decode_step(self.handle, mode, steps, ctypes.addressof(buf), self.stats)
        else:
            c = list(cands) if cands is not None else [0]
            o = DecodeOpts(mode, NDIFF_SAMPLER_THRESHOLD if tau is not None else NDIFF_SAMPLER_TOPK,
                           steps, 0.0 if tau is None else tau, tau_revise, len(c),
                           (ctypes.c_int * 2)(*(c + c)[:2]))
            n = ndiff_decode_step_ex(self.handle, o, ctypes.addressof(buf), self.stats)
        return list(buf[:n])

    def generate(self, mode: int, n_new: int, steps: int = 1, tau: float | None = None,
                 tau_revise: float = 2.0, cands=None):
        out = []
        while len(out) < n_new:
            out.extend(self.step(mode, steps, tau, tau_revise, cands))
        return out[:n_new]

    # ---- batched sessions (batch > 1)
    def prefill_batch(self, prompts):
        """prompts: a list of B token lists (ragged lengths)."""
        import numpy as np
        lens = np.ascontiguousarray(np.array([len(p) for p in prompts], dtype=np.int32))
        flat = np.ascontiguousarray(np.concatenate([np.asarray(p, dtype=np.int32) for p in prompts]))
        _call("ndiff_prefill_batch", self.handle, flat.ctypes.data, lens.ctypes.data,
              _stream(None))

    def step_batch(self, mode: int, steps: int = 1, tau: float | None = None,
                   tau_revise: float = 2.0):
        """One decode cycle of every sequence: a list of B token lists."""
        B = self.batch
        buf = (ctypes.c_int32 * (32 * B))()
        n = (ctypes.c_int32 * B)()
        o = DecodeOpts(mode, NDIFF_SAMPLER_TOPK if tau is None else NDIFF_SAMPLER_THRESHOLD, steps,
                       0.0 if tau is None else tau, tau_revise)
        _call("ndiff_decode_step_batch", self.handle, ctypes.byref(o), ctypes.addressof(buf),
              ctypes.addressof(n), ctypes.byref(self.stats), _stream(None))
        return [list(buf[32 * b: 32 * b + n[b]]) for b in range(B)]

    def generate_batch(self, mode: int, n_new: int, steps: int = 1, tau: float | None = None,
                       tau_revise: float = 2.0):
        out = [[] for _ in range(self.batch)]
        while min(len(o) for o in out) < n_new:
            for o, t in zip(out, self.step_batch(mode, steps, tau, tau_revise)):
                o.extend(t)
        return [o[:n_new] for o in out]

    def state_batch(self):
        B = self.batch
        kv = (ctypes.c_int32 * B)()
        last = (ctypes.c_int32 * B)()
        _call("ndiff_model_state_batch", self.handle, ctypes.addressof(kv), ctypes.addressof(last))
        return list(kv), list(last)

    def forward(self, ids, mode: int):
        import numpy as np
        arr = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
        T = int(arr.shape[0])
        logits = np.empty((T, self.vocab), dtype=np.float32)
        ndiff_model_forward(self.handle, arr.ctypes.data, T, mode, logits.ctypes.data)
        return logits

    def state(self):
        return ndiff_model_state(self.handle)

    def read_weight(self, tensor_id: int, offset: int, count: int):
        import numpy as np
        out = np.empty(count, dtype=np.float32)
        ndiff_model_read_weight(self.handle, tensor_id, offset, count, out.ctypes.data)
        return out
