#!/usr/bin/env python3
"""Benchmark of the decode-step hot path on B300 (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Workloads (seeded synthetic inputs, shapes of the 8B-like configurations):
  attn-batched  one decode-step pass over a batch of 64 sequences with KV
                prefixes uniform in [512, 8192]: block-causal attention
                (32 query / 8 KV heads x 128, 32-token block), logits
                reduction over 64 x 32 x 151936 bf16 logits, unmask (k = 8) and
                verify/accept. value = algorithmic HBM bytes of the pass / time.
  attn-single   block attention alone, batch 1, prefix 4096 (17 MB of KV,
                rotated over copies so every launch reads from HBM).
  attn-long     block attention alone, batch 4, prefix 32768.

Every run also decodes with the 8B-shaped random-init model (36 layers,
d_model 4096, 32/8 heads x 128, SwiGLU 12288, vocab 151936, bf16 weights; batch
1, 1024-token prompt) unless --model-tokens 0: AR, temperature-0
self-speculation (32-token diffusion drafts, one drafting forward) and fused
self-speculation (one forward verifies a block and drafts the next) each
generate --model-tokens tokens through the C ABI's decode step; reported as
tokens/s, tokens per forward and whether the self-speculation tokens equal
the AR tokens. A labelled forced-acceptance run (the same body with a two-id
vocabulary, so every draft is accepted) shows the machinery's L = 32 ceiling.

Unless --batch-model 0, the same 8B-shaped model also decodes a batch of 64
sequences together (ragged prompts uniform in [512, 2048] tokens; every
projection on the wide tensor-core kernel over 64 x 32 token rows): AR and
self-speculation, --batch-tokens tokens per sequence, reported as tokens/s of
the whole batch, tokens per batch forward and the forward's tensor FLOP rate.

Under torchrun (N > 1) each rank runs an independent replica of the workload
(sequences are independent: no collective on the data path); value is the
work of all ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "block-attn HBM GB/s (% of peak); self-spec tokens/s and tokens/forward at 8B"
# DRAM bytes (read + write) of one attention launch and its split merge, from
# ncu captures of the current kernels on these workloads (summary under
# profiles/); None where no capture exists.
ATTN_TRAFFIC = {"attn-batched": 1016270592 + 1821696,
                "attn-long": 539068672 + 389120 + 8535808,
                "attn-single": 17227008 + 0 + 9068032}
SPEC_HBM_GBS = 8000.0
L2_BYTES = 126e6


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    return 6400.0, 1800.0, 1400.0, "fallback"


# --------------------------------------------------------------------------
# clocks sampled during the timed region
# --------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        rows = [r for r in self.rows if len(r) > 8]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [v for v in (num(r[1]) for r in rows) if v is not None]
        mx = [v for v in (num(r[2]) for r in rows) if v is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------
def attn_bytes(lengths, T, Hq, Hkv, D):
    """Algorithmic bytes of one attention launch: every visible K and V row
    once (Hkv x D bf16 each), Q read and O written once."""
    kv = int(np.sum(np.asarray(lengths, dtype=np.int64) + T)) * Hkv * D * 2 * 2
    qo = len(lengths) * T * Hq * D * 2 * 2
    return kv + qo


class AttnWorkload:
    """Attention-only or full batched pass on device-resident inputs."""

    def __init__(self, name, rank, host_only=False):
        import torch
        from self_speculative_lm_block_b300 import synth
        if host_only:
            nd = None
        else:
            from self_speculative_lm_block_b300 import ndiff as nd
        self.nd, self.torch = nd, torch
        self.name = name
        c = {"attn-single": synth.ATTN_SINGLE, "attn-batched": synth.ATTN_BATCHED,
             "attn-long": synth.ATTN_LONG}[name]
        self.c = c
        seed = c["seed"] + 1000 * rank
        lengths = synth.attn_lengths(c["B"], seed, c["P_lo"], c["P_hi"])
        self.lengths = lengths
        self.Lmax = int(c["P_hi"]) + c["T"]
        inp = synth.attn_inputs(c["B"], c["T"], c["Hq"], c["Hkv"], c["D"], lengths, self.Lmax, seed)
        self.host = inp
        self.name, self.c = name, c
        self.full = name == "attn-batched"
        self.scale = inp.scale
        if host_only:
            self.attn_bytes = attn_bytes(lengths, c["T"], c["Hq"], c["Hkv"], c["D"])
            if self.full:
                self.V = c["V"]
                self.logits_host = synth.logits(64, self.V, c["logit_sigma"], seed)
            self.ncopy = 1
            return
        dev = "cuda"
        self.q = inp.q.to(dev)
        self.kv_len = inp.kv_len.to(dev)
        self.scale = inp.scale
        # rotate over copies when one copy would stay resident in L2
        one = inp.k_cache.numel() * 2 * 2
        self.ncopy = 1 if one >= 4 * L2_BYTES else int(np.ceil(4 * L2_BYTES / one))
        self.k = [inp.k_cache.to(dev) for _ in range(self.ncopy)]
        self.v = [inp.v_cache.to(dev) for _ in range(self.ncopy)]
        self.out = torch.empty_like(self.q)
        B, T, Hq, Hkv, D = c["B"], c["T"], c["Hq"], c["Hkv"], c["D"]
        self.ws_bytes = nd.ndiff_block_attn_workspace_size(nd.NDIFF_BF16, B, T, Hq, Hkv, D, self.Lmax)
        self.ws = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8, device=dev)
        self.attn_bytes = attn_bytes(lengths, T, Hq, Hkv, D)
        self.step_bytes = self.attn_bytes
        self.full = name == "attn-batched"
        self.attn_launches = 1 + (1 if self.ws_bytes > 0 else 0)
        self.launches = self.attn_launches
        if self.full:
            V = c["V"]
            R = B * T
            self.V, self.R = V, R
            self.logits = synth.logits(R, V, c["logit_sigma"], seed).to(dev)
            draft, target, _ = synth.draft_target(B, T, V, seed)
            self.draft = draft.to(dev)
            self.ids = torch.empty(R, dtype=torch.int32, device=dev)
            self.conf = torch.empty(R, dtype=torch.float32, device=dev)
            self.L = torch.empty(B, dtype=torch.int32, device=dev)
            self.n = torch.empty(B, dtype=torch.int32, device=dev)
            self.commit = torch.empty((B, T), dtype=torch.int32, device=dev)
            _, _, mask = synth.unmask_inputs(B, T, V, seed, all_masked=True)
            self.u_mask0 = mask.to(dev)
            self.u_mask = self.u_mask0.clone()
            self.blk = torch.zeros((B, T), dtype=torch.int32, device=dev)
            self.drf = torch.full((B, T), -1, dtype=torch.int32, device=dev)
            self.chosen = torch.empty((B, 8), dtype=torch.int32, device=dev)
            # logits read; ids/conf written; unmask and accept read/write [B][T] ints
            self.step_bytes += R * V * 2 + R * 8 + B * T * 4 * 10
            self.launches += 3
        self.i = 0

    def step(self, attn_only=False):
        nd = self.nd
        c = self.c
        j = self.i % self.ncopy
        self.i += 1
        nd.ndiff_block_attn(nd.NDIFF_BF16, self.q, self.k[j], self.v[j], self.kv_len, c["B"], c["T"],
                            c["Hq"], c["Hkv"], c["D"], self.Lmax, nd.NDIFF_CAUSAL, self.scale,
                            self.out, self.ws, self.ws_bytes)
        if self.full and not attn_only:
            nd.ndiff_logits_reduce(nd.NDIFF_BF16, self.logits, self.R, self.V, self.V, self.V - 1,
                                   self.ids, self.conf)
            nd.ndiff_verify_accept(self.draft, self.ids, c["B"], c["T"], self.L, self.commit, self.n,
                                   None)
            self.u_mask.copy_(self.u_mask0)
            nd.ndiff_unmask(self.conf, self.ids, c["B"], c["T"], 8, self.u_mask, self.blk, self.drf,
                            self.chosen)

    def e2e_step(self, pinned):
        """Host buffers in, host results out, through the C ABI."""
        nd = self.nd
        c = self.c
        self.q.copy_(pinned["q"], non_blocking=True)
        self.k[0].copy_(pinned["k"], non_blocking=True)
        self.v[0].copy_(pinned["v"], non_blocking=True)
        self.kv_len.copy_(pinned["kv_len"], non_blocking=True)
        nd.ndiff_block_attn(nd.NDIFF_BF16, self.q, self.k[0], self.v[0], self.kv_len, c["B"], c["T"],
                            c["Hq"], c["Hkv"], c["D"], self.Lmax, nd.NDIFF_CAUSAL, self.scale,
                            self.out, self.ws, self.ws_bytes)
        pinned["out"].copy_(self.out, non_blocking=True)
        h2d = sum(pinned[x].numel() * pinned[x].element_size() for x in ("q", "k", "v", "kv_len"))
        d2h = pinned["out"].numel() * 2
        if self.full:
            self.logits.copy_(pinned["logits"], non_blocking=True)
            self.draft.copy_(pinned["draft"], non_blocking=True)
            nd.ndiff_logits_reduce(nd.NDIFF_BF16, self.logits, self.R, self.V, self.V, self.V - 1,
                                   self.ids, self.conf)
            nd.ndiff_verify_accept(self.draft, self.ids, c["B"], c["T"], self.L, self.commit, self.n,
                                   None)
            pinned["commit"].copy_(self.commit, non_blocking=True)
            h2d += pinned["logits"].numel() * 2 + pinned["draft"].numel() * 4
            d2h += pinned["commit"].numel() * 4
        return h2d, d2h

    def pinned(self):
        torch = self.torch
        d = {"q": self.host.q.pin_memory(), "k": self.host.k_cache.pin_memory(),
             "v": self.host.v_cache.pin_memory(), "kv_len": self.host.kv_len.pin_memory(),
             "out": torch.empty(self.q.shape, dtype=self.q.dtype).pin_memory()}
        if self.full:
            d["logits"] = self.logits.cpu().pin_memory()
            d["draft"] = self.draft.cpu().pin_memory()
            d["commit"] = torch.empty(self.commit.shape, dtype=torch.int32).pin_memory()
        return d

    def config(self):
        c = self.c
        cfg = {"workload": self.name, "batch": c["B"], "q_heads": c["Hq"], "kv_heads": c["Hkv"],
               "head_dim": c["D"], "block": c["T"],
               "kv_prefix": [int(c["P_lo"]), int(c["P_hi"])], "mask": "causal",
               "l2": ("inputs larger than L2" if self.ncopy == 1 else
                      f"rotating {self.ncopy} KV copies (> 4x L2)")}
        if self.full:
            cfg.update({"vocab": self.V, "logits": "bf16 N(0,4^2)", "unmask_k": 8})
        return cfg

    def oracle_sample(self):
        """Oracle time on a bounded sample of the same pass -> GB/s of that sample."""
        from oracle import attention as OA
        from oracle import decode as OD
        h = self.host
        B = 2 if self.name != "attn-long" else 1
        q = h.q[:B].float().numpy()
        P = h.kv_len[:B].numpy()
        Lm = int(P.max()) + self.c["T"]
        k = h.k_cache[:B, :, :Lm].float().numpy()
        v = h.v_cache[:B, :, :Lm].float().numpy()
        t0 = time.perf_counter()
        OA.block_attn(q, k, v, P, OA.CAUSAL, self.scale)
        nbytes = attn_bytes(P, self.c["T"], self.c["Hq"], self.c["Hkv"], self.c["D"])
        desc = f"{B} sequence(s) of the attention"
        if self.full:
            rows = 64
            src = self.logits_host if self.nd is None else self.logits[:rows].cpu()
            x = src.float().numpy()
            OD.logits_reduce(x, exclude_id=self.V - 1)
            nbytes += rows * self.V * 2
            desc += f" + {rows} logits rows"
        dt = time.perf_counter() - t0
        return nbytes / dt / 1e9, desc, dt


def host_cpu():
    """The host the oracle is timed on: its CPU model (from /proc/cpuinfo) and
    the number of cores this process may run on (nproc)."""
    model = "unknown"
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    try:
        nproc = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        nproc = os.cpu_count()
    return {"model": model, "nproc": nproc}


_ONE_THREAD_ENV = {"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1",
                   "BLIS_NUM_THREADS": "1", "NUMEXPR_NUM_THREADS": "1"}


def oracle_sample_1thread(name):
    """The oracle's sample of workload `name` timed on one core (the plain
    single-threaded CPU baseline): NumPy's BLAS and OpenMP pools limited to
    one thread, by threadpoolctl where it is installed, else in a child
    process started with the thread-count variables set to 1 (the pools are
    sized when NumPy loads). Returns (GB/s, description, seconds, threads)."""
    try:
        import threadpoolctl
    except ImportError:
        threadpoolctl = None
    if threadpoolctl is not None:
        wl = AttnWorkload(name, 0, host_only=True)
        with threadpoolctl.threadpool_limits(limits=1):
            used = max([i.get("num_threads", 1) for i in threadpoolctl.threadpool_info()] or [1])
            v, desc, dt = wl.oracle_sample()
        return v, desc, dt, used
    env = dict(os.environ, **_ONE_THREAD_ENV)
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-sample-only",
                        "--workload", name], env=env, capture_output=True, text=True, timeout=900)
    if r.returncode != 0:
        raise RuntimeError("oracle sample failed: " + r.stderr[-2000:])
    d = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])
    return d["value"], d["sample"], d["seconds"], 1


def weight_bytes_8b(c):
    d, D, Hq, Hkv, f, V = c["d_model"], c["head_dim"], c["n_heads"], c["n_kv_heads"], c["ffn"], c["vocab"]
    per_layer = ((Hq + 2 * Hkv) * D * d + d * Hq * D + 2 * f * d + d * f) * 2
    return c["layers"] * per_layer + V * d * 2


def run_model(rank, n_tokens, steps=1):
    """AR and self-speculative decoding of the 8B-shaped model on this rank."""
    import torch
    from self_speculative_lm_block_b300 import ndiff as nd
    from self_speculative_lm_block_b300 import synth
    c = synth.MODEL_8B
    seed = c["seed"] + 1000 * rank
    m = nd.Model(c["layers"], c["d_model"], c["n_heads"], c["n_kv_heads"], c["head_dim"], c["ffn"],
                 c["vocab"], dtype="bf16", max_seq=c["prompt"] + n_tokens + 512, seed=seed)
    prompt = synth.prompt(c["prompt"], c["vocab"], seed)
    out = {"model": "8B-shaped random init (36L, d4096, 32/8x128, ffn 12288, V151936, bf16)",
           "prompt": c["prompt"], "tokens": n_tokens}
    res = {}
    for name, mode in (("ar", nd.NDIFF_MODE_AR), ("selfspec", nd.NDIFF_MODE_SELFSPEC),
                       ("selfspec_fused", nd.NDIFF_MODE_SELFSPEC_FUSED)):
        m.prefill(prompt)
        m.step(mode, steps)                      # warm-up cycle (graph capture)
        m.prefill(prompt)
        m.stats = nd.Stats()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        toks = m.generate(mode, n_tokens, steps)
        dt = time.perf_counter() - t0
        st = m.stats
        res[name] = toks
        out[name] = {"tokens_per_s": st.tokens / dt, "forwards": int(st.forwards),
                     "tokens_per_forward": st.tokens / st.forwards,
                     "ms_per_forward": dt * 1e3 / st.forwards, "seconds": dt}
        if name.startswith("selfspec"):
            hist = [int(x) for x in st.accept_hist]
            out[name]["accept_len_hist"] = {str(i): v for i, v in enumerate(hist) if v}
            out[name]["draft_forwards_per_block"] = steps
    # quadratic self-speculation: the verifying forward also drafts the next
    # block for the two acceptance lengths below 32 that the linear run saw
    # most often (ties: the shorter)
    hist = out["selfspec"].get("accept_len_hist", {})
    ranked = sorted(((-v, int(k)) for k, v in hist.items() if int(k) < 32))
    cands = [k for _, k in ranked[:2]] or [0]
    if len(cands) == 1:
        cands.append(1 if cands[0] != 1 else 0)
    m.prefill(prompt)
    m.step(nd.NDIFF_MODE_SELFSPEC_QUAD, cands=cands)   # warm-up (graph capture)
    m.prefill(prompt)
    m.stats = nd.Stats()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    toks = m.generate(nd.NDIFF_MODE_SELFSPEC_QUAD, n_tokens, cands=cands)
    dt = time.perf_counter() - t0
    st = m.stats
    qh = [int(x) for x in st.accept_hist]
    out["selfspec_quadratic"] = {
        "candidates": cands, "tokens_per_s": st.tokens / dt, "forwards": int(st.forwards),
        "tokens_per_forward": st.tokens / st.forwards, "ms_per_forward": dt * 1e3 / st.forwards,
        "seconds": dt, "accept_len_hist": {str(i): v for i, v in enumerate(qh) if v},
        "rows_per_forward": 128, "equals_ar": toks == res["ar"]}
    # drafting forwards per block (steps S; each unmasks 32/S slots)
    sweep = {}
    for S in (2, 4):
        ns = min(n_tokens, 64)
        m.prefill(prompt)
        m.step(nd.NDIFF_MODE_SELFSPEC, S)
        m.prefill(prompt)
        m.stats = nd.Stats()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        toks = m.generate(nd.NDIFF_MODE_SELFSPEC, ns, S)
        dt = time.perf_counter() - t0
        st = m.stats
        sweep[str(S)] = {"tokens": ns, "tokens_per_s": st.tokens / dt, "forwards": int(st.forwards),
                         "tokens_per_forward": st.tokens / st.forwards,
                         "ms_per_forward": dt * 1e3 / st.forwards,
                         "equals_ar": toks == res["ar"][:len(toks)]}
    out["selfspec_steps_sweep"] = sweep
    # the threshold sampler's host-driven round loop (a 4-byte read between
    # rounds), at tau = 0: one drafting round per block, the same forwards as
    # the one-round top-k draft above, so the difference is the loop's cost
    m.prefill(prompt)
    m.step(nd.NDIFF_MODE_SELFSPEC, 1, tau=0.0)
    m.prefill(prompt)
    m.stats = nd.Stats()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    toks = m.generate(nd.NDIFF_MODE_SELFSPEC, min(n_tokens, 64), 1, tau=0.0)
    dt = time.perf_counter() - t0
    st = m.stats
    out["selfspec_threshold_tau0"] = {"tokens_per_s": st.tokens / dt, "forwards": int(st.forwards),
                                      "ms_per_forward": dt * 1e3 / st.forwards,
                                      "equals_ar": toks == res["ar"][:len(toks)]}
    wb = weight_bytes_8b(c)
    out["weight_bytes_per_forward"] = wb
    out["ar"]["weight_stream_gbs"] = wb / (out["ar"]["ms_per_forward"] * 1e-3) / 1e9
    out["selfspec_equals_ar"] = res["selfspec"] == res["ar"]
    out["selfspec_fused_equals_ar"] = res["selfspec_fused"] == res["ar"]
    out["note"] = ("random-init weights: tokens per forward is not the trained model's; "
                   "decode steps are host-synchronous calls (host buffers in and out)")
    m.close()
    return out


def run_lm_head(reps=20):
    """The 8B LM head (151936 x 4096 bf16, 1.24 GB: larger than L2) at a
    32-token block and at one token: the fused argmax/confidence epilogue
    against the GEMM that stores fp32 logits followed by the reduce kernel.
    Device-timed CUDA-graph replays of `reps` calls each."""
    import torch
    from self_speculative_lm_block_b300 import ndiff as nd
    from self_speculative_lm_block_b300 import synth
    V, d = synth.MODEL_8B["vocab"], synth.MODEL_8B["d_model"]
    gen = torch.Generator(device="cuda").manual_seed(1005)
    w = (torch.randn((V, d), device="cuda", generator=gen) * 0.02).to(torch.bfloat16)
    out = {"shape": f"{V} x {d} bf16", "weight_bytes": V * d * 2}
    s = torch.cuda.Stream()

    def time_graph(fn):
        with torch.cuda.stream(s):
            fn()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for _ in range(reps):
                    fn()
            g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            g.replay()                       # replays on the current stream: s
            e1.record(s)
            torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / reps

    for M in (1, 32):
        x = torch.randn((M, d), device="cuda", generator=gen).to(torch.bfloat16)
        ids = torch.empty(M, dtype=torch.int32, device="cuda")
        conf = torch.empty(M, dtype=torch.float32, device="cuda")
        need_f = nd.ndiff_lm_head_argmax_workspace_size(M, V, d)
        ws_f = torch.empty(need_f, dtype=torch.uint8, device="cuda")
        y = torch.empty((M, V), dtype=torch.float32, device="cuda")
        need_g = nd.ndiff_gemm_bf16_workspace_size(M, V, d)
        ws_g = torch.empty(max(need_g, 16), dtype=torch.uint8, device="cuda")
        st = s.cuda_stream

        def fused():
            nd.ndiff_lm_head_argmax(x, w, M, V, d, V - 1, ids, conf, ws_f, need_f, st)

        def unfused():
            nd.ndiff_gemm_bf16(x, w, M, V, d, y, V, ws_g, need_g, st)
            nd.ndiff_logits_reduce(nd.NDIFF_F32, y, M, V, V, V - 1, ids, conf, st)

        tf, tu = time_graph(fused), time_graph(unfused)
        out[f"tokens_{M}"] = {"fused_us": tf, "unfused_us": tu,
                              "fused_weight_gbs": V * d * 2 / (tf * 1e-6) / 1e9}
    return out


def run_select_batch(B=65536, T=32, k=8, usets=48, vsets=8):
    """Unmask (top-k) and verify/accept over a batch large enough for a
    bandwidth figure: 65536 sequences of 32 slots. Every launch in the timed
    graph works on its own copy of the inputs (unmask: 48 copies of 34 MB, one
    per launch, mask words reset before the replay and outside the timed
    region; verify: 8 copies of 26 MB cycled), so each launch reads its inputs
    from HBM rather than from the 126 MB L2. Algorithmic bytes per sequence:
    unmask reads conf, pred and the mask word and writes the mask word, the k
    chosen slots and k draft and next-input tokens; verify reads draft and
    target and writes the commit row, accept length and commit count, and
    reads and writes the prefix length."""
    import torch
    from self_speculative_lm_block_b300 import ndiff as nd
    from self_speculative_lm_block_b300 import synth
    hbm, _, _, src = _peaks()
    conf, pred, mask = synth.unmask_inputs(B, T, 151936, 4001)
    draft, target, _ = synth.draft_target(B, T, 151936, 4002)
    conf, pred, mask, draft, target = (t.cuda() for t in (conf, pred, mask, draft, target))
    z = lambda *shape: torch.zeros(shape, dtype=torch.int32, device="cuda")
    U = [dict(conf=conf.clone(), pred=pred.clone(), mk=mask.clone(), blk=z(B, T), dr=z(B, T),
              ch=z(B, k)) for _ in range(usets)]
    V = [dict(draft=draft.clone(), target=target.clone(), L=z(B), n=z(B), com=z(B, T), kv=z(B))
         for _ in range(vsets)]
    s = torch.cuda.Stream()

    def time_graph(fn, reps, nsets, reset=lambda: None):
        with torch.cuda.stream(s):
            reset()
            for i in range(nsets):
                fn(i)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for r in range(reps):
                    fn(r % nsets)
            reset()
            g.replay()
            torch.cuda.synchronize()
            reset()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            g.replay()
            e1.record(s)
            torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / reps

    def reset_masks():
        for u in U:
            u["mk"].copy_(mask)

    def unmask(i):
        u = U[i]
        nd.ndiff_unmask(u["conf"], u["pred"], B, T, k, u["mk"], u["blk"], u["dr"], u["ch"],
                        s.cuda_stream)

    def verify(i):
        v = V[i]
        nd.ndiff_verify_accept(v["draft"], v["target"], B, T, v["L"], v["com"], v["n"], v["kv"],
                               s.cuda_stream)

    t_u = time_graph(unmask, usets, usets, reset_masks)
    t_v = time_graph(verify, 48, vsets)
    bytes_u = B * (T * 4 * 2 + 4 + 4 + k * 4 * 3)
    bytes_v = B * (T * 4 * 3 + 4 * 4)
    res = {"label": f"{B} sequences x {T} slots, every launch on its own copy of the inputs "
                    "(throughput figure; decode steps use a few sequences)"}
    for name, t, nb in (("unmask_k8", t_u, bytes_u), ("verify_accept", t_v, bytes_v)):
        gbs = nb / (t * 1e-6) / 1e9
        res[name] = {"us": t, "bytes": nb, "gbs": gbs, "frac_hbm": gbs / hbm, "peak_source": src}
    return res


def run_forced_accept(rank, n_tokens=256):
    """The fused self-speculation machinery with every draft accepted: the
    8B-shaped body with a two-id vocabulary ([MASK] and one token), so each
    fused forward commits 32 tokens. Labelled as the L = 32 ceiling of the
    machinery; the LM head is 2 ids instead of 151936."""
    import torch
    from self_speculative_lm_block_b300 import ndiff as nd
    from self_speculative_lm_block_b300 import synth
    c = synth.MODEL_8B
    m = nd.Model(c["layers"], c["d_model"], c["n_heads"], c["n_kv_heads"], c["head_dim"], c["ffn"],
                 2, dtype="bf16", max_seq=1024 + n_tokens + 96, seed=c["seed"] + 1000 * rank)
    m.prefill([0] * 1024)
    m.step(nd.NDIFF_MODE_SELFSPEC_FUSED)
    m.prefill([0] * 1024)
    m.stats = nd.Stats()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    m.generate(nd.NDIFF_MODE_SELFSPEC_FUSED, n_tokens)
    dt = time.perf_counter() - t0
    st = m.stats
    out = {"label": "L = 32 machinery ceiling (vocabulary of 2: every draft accepted)",
           "tokens_per_s": st.tokens / dt, "forwards": int(st.forwards),
           "tokens_per_forward": st.tokens / st.forwards, "ms_per_forward": dt * 1e3 / st.forwards}
    m.close()
    return out


def run_model_batched(rank, B, n_tokens):
    """AR and self-speculative decoding of B ragged sequences together."""
    import numpy as np
    import torch
    from self_speculative_lm_block_b300 import ndiff as nd
    from self_speculative_lm_block_b300 import synth
    c = synth.MODEL_8B
    seed = c["seed"] + 1000 * rank
    lengths = [int(x) for x in np.random.default_rng(seed).integers(512, 2049, size=B)]
    prompts = [list(synth.prompt(n, c["vocab"], seed + i)) for i, n in enumerate(lengths)]
    m = nd.Model(c["layers"], c["d_model"], c["n_heads"], c["n_kv_heads"], c["head_dim"], c["ffn"],
                 c["vocab"], dtype="bf16", max_seq=max(lengths) + 32 * n_tokens + 64, seed=seed,
                 batch=B)
    out = {"batch": B, "prompt_lengths": "uniform in [512, 2048]", "tokens_per_sequence": n_tokens}
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    m.prefill_batch(prompts)
    out["prefill_s"] = time.perf_counter() - t0
    out["prefill_tokens"] = int(sum(lengths) - B)
    res = {}
    for name, mode in (("ar", nd.NDIFF_MODE_AR), ("selfspec", nd.NDIFF_MODE_SELFSPEC)):
        m.prefill_batch(prompts)
        m.step_batch(mode, 1)                    # warm-up cycle (graph capture)
        m.prefill_batch(prompts)
        m.stats = nd.Stats()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        toks = m.generate_batch(mode, n_tokens, 1)
        dt = time.perf_counter() - t0
        st = m.stats
        res[name] = toks
        out[name] = {"tokens_per_s": st.tokens / dt, "forwards": int(st.forwards),
                     "tokens_per_forward": st.tokens / st.forwards,
                     "ms_per_forward": dt * 1e3 / st.forwards, "seconds": dt}
    # a block forward multiplies 64 x 32 token rows with every weight once
    flops = 2.0 * B * 32 * (weight_bytes_8b(c) / 2)
    out["selfspec"]["block_forward_tflops"] = flops / (out["selfspec"]["ms_per_forward"] * 1e-3) / 1e12
    out["selfspec_equals_ar"] = all(a == b for a, b in zip(res["selfspec"], res["ar"]))
    m.close()
    return out


def make_workload(name, rank):
    if name.startswith("attn-"):
        return AttnWorkload(name, rank)
    raise SystemExit(f"unknown workload {name}")


def run_reference(args, rank, world):
    """The oracle as it stands, on the host cores, each step a bounded sample."""
    if rank != 0:
        return
    wl = AttnWorkload(args.workload, 0, host_only=True)
    vals, secs, desc = [], [], ""
    for i in range(args.warmup + args.steps):
        v, desc, dt, threads = oracle_sample_1thread(args.workload)
        if i >= args.warmup:
            vals.append(v)
            secs.append(dt)
    value = float(np.mean(vals))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": float(np.mean(secs)) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": wl.config(),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads,
                             "kind": "oracle", "sample": desc, "host": host_cpu()},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def reduce_over_ranks(x: float, op: str, world: int, device) -> float:
    """A per-rank number combined over the replicas: "max" (the slowest
    rank's time, which bounds the job) or "sum" (all ranks' throughput)."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([x], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(
        t, op=torch.distributed.ReduceOp.MAX if op == "max" else torch.distributed.ReduceOp.SUM)
    return float(t.item())


def job_gbs(step_bytes: int, world: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every replica processes step_bytes per step, the job
    takes the slowest replica's time."""
    return step_bytes * world / (ms_per_step * 1e-3) / 1e9


def run_attn_alone(name, rank, steps, warmup):
    """Block attention of workload `name` (attn-single: batch 1 x 4096 keys;
    attn-long: batch 4 x 32768 keys) timed alone: CUDA-graph replays of its
    launches on device-resident inputs, rotating over KV copies when one copy
    would stay in L2. Returns its roofline block (achieved = algorithmic bytes
    per launch / device time per launch)."""
    import torch
    wl = AttnWorkload(name, rank)
    for _ in range(warmup):
        wl.step(attn_only=True)
    torch.cuda.synchronize()
    g = capture(torch, lambda: wl.step(attn_only=True), wl.ncopy)
    reps = max(2, (steps + wl.ncopy - 1) // wl.ncopy)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (reps * wl.ncopy)
    gbs = wl.attn_bytes / (ms * 1e-3) / 1e9
    hbm, _, _, src = _peaks()
    out = {"config": wl.config(), "kernel": "attn_bf16_kernel (+attn_combine_kernel)", "bound": "hbm",
           "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm, "peak_source": src,
           "frac_of_spec_8tbs": gbs / SPEC_HBM_GBS, "bytes_per_launch": wl.attn_bytes,
           "ms_per_launch": ms, "traffic": ATTN_TRAFFIC.get(name), "launches": reps * wl.ncopy}
    del wl, g
    torch.cuda.empty_cache()
    return out


def capture(torch, fn, n):
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for _ in range(n):
                fn()
    torch.cuda.current_stream().wait_stream(s)
    return g


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="attn-batched",
                    choices=["attn-batched", "attn-single", "attn-long"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--model-tokens", type=int, default=512,
                    help="tokens generated per mode by the 8B-shaped model (0: skip)")
    ap.add_argument("--batch-model", type=int, default=64,
                    help="sequences of the batched 8B-shaped decode (0: skip)")
    ap.add_argument("--batch-tokens", type=int, default=32,
                    help="tokens generated per sequence and mode by the batched decode")
    ap.add_argument("--oracle-sample-only", action="store_true",
                    help="(internal) print one oracle sample of --workload as JSON and exit")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.oracle_sample_only:
        v, desc, dt = AttnWorkload(args.workload, 0, host_only=True).oracle_sample()
        print(json.dumps({"value": v, "sample": desc, "seconds": dt}), flush=True)
        return

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    wl = make_workload(args.workload, rank)
    for _ in range(args.warmup):
        wl.step()
    barrier()
    # The timed region replays CUDA graphs of whole steps, so that host launch
    # overhead stays out of the device timeline of the small configurations.
    per_graph = wl.ncopy
    g_step = capture(torch, wl.step, per_graph)
    g_attn = capture(torch, lambda: wl.step(attn_only=True), per_graph)
    reps = max(1, (args.steps + per_graph - 1) // per_graph)
    for _ in range(2):
        g_step.replay()
        g_attn.replay()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        e0.record()
        for _ in range(reps):
            g_step.replay()
        e1.record()
        barrier()
        a0.record()
        for _ in range(reps):
            g_attn.replay()
        a1.record()
        barrier()
    steps_done = reps * per_graph
    ms_total = reduce_over_ranks(e0.elapsed_time(e1), "max", world, "cuda")
    ms_step = ms_total / steps_done
    value = job_gbs(wl.step_bytes, world, ms_step)
    attn_ms = a0.elapsed_time(a1) / steps_done
    attn_gbs = wl.attn_bytes / (attn_ms * 1e-3) / 1e9

    # end to end through the C ABI with pinned host buffers
    pinned = wl.pinned()
    for _ in range(2):
        wl.e2e_step(pinned)
    barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_e2e = max(2, min(args.steps, 5))
    f0.record()
    for _ in range(n_e2e):
        h2d, d2h = wl.e2e_step(pinned)
    f1.record()
    barrier()
    e2e_ms = reduce_over_ranks(f0.elapsed_time(f1), "max", world, "cuda") / n_e2e
    e2e_val = job_gbs(wl.step_bytes, world, e2e_ms)

    # the other attention configurations (batch 1 x 4096, batch 4 x 32768)
    extra_attn = {}
    if args.workload == "attn-batched":
        for nm in ("attn-single", "attn-long"):
            extra_attn[nm.replace("-", "_")] = run_attn_alone(nm, rank, args.steps, args.warmup)

    model = run_model(rank, args.model_tokens) if args.model_tokens > 0 else None
    lm_head = run_lm_head() if args.model_tokens > 0 else None
    forced = run_forced_accept(rank) if args.model_tokens > 0 else None
    select = run_select_batch()
    batched = run_model_batched(rank, args.batch_model, args.batch_tokens) \
        if args.batch_model > 0 else None
    if model is not None and world > 1:
        for k in ("ar", "selfspec", "selfspec_fused"):
            model[k]["tokens_per_s_all_ranks"] = reduce_over_ranks(model[k]["tokens_per_s"], "sum",
                                                                   world, "cuda")

    hbm, _, _, src = _peaks()
    if rank == 0:
        out = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
               "steps": steps_done, "warmup": args.warmup, "ms_per_step": ms_step,
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
               "data": "synthetic", "config": wl.config(),
               "roofline": {"kernel": "attn_bf16_kernel (+attn_combine_kernel)", "bound": "hbm",
                            "achieved": attn_gbs, "peak": hbm, "unit": "GB/s",
                            "frac": attn_gbs / hbm, "peak_source": src,
                            "frac_of_spec_8tbs": attn_gbs / SPEC_HBM_GBS,
                            "bytes_per_launch": wl.attn_bytes, "ms_per_launch": attn_ms,
                            "traffic": ATTN_TRAFFIC.get(args.workload)},
               "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
               "gpu_launches": wl.launches * steps_done,
               "timing": "CUDA-graph replay of whole steps; attention timed by a graph of its launches",
               "clocks": clk.summary()}
        out.update(extra_attn)
        if model is not None:
            out["model_8b"] = model
        if lm_head is not None:
            out["lm_head_8b"] = lm_head
        if forced is not None:
            out["model_8b"]["forced_accept_fused"] = forced
        out["select_65536"] = select
        if batched is not None:
            out["model_8b_batched"] = batched
        if not args.no_cpu_baseline:
            cv, desc, dt, threads = oracle_sample_1thread(args.workload)
            out["cpu_baseline"] = {"value": cv, "unit": "GB/s", "cores": threads,
                                   "kind": "oracle", "sample": desc, "seconds": dt,
                                   "host": host_cpu()}
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
