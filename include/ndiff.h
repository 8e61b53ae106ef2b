/*
 * ndiff.h — C ABI of libndiff: the decode step over a 32-token block of a
 * tri-mode (autoregressive / block-wise diffusion / self-speculation) language
 * model, for one NVIDIA B300 (sm_103a).
 *
 * Sources of the operations (page title, then section):
 *   [TRI]  "Nemotron-Labs-Diffusion: A Tri-Mode Language Model Unifying
 *          Autoregressive, Diffusion, and Self-Speculation Decoding"
 *          (hotpaper.ai): Abstract; "기술적 접근법 / 모듈" (technical approach /
 *          modules: block-wise attention).
 *   [FFI]  "NVIDIA 发布 Nemotron-Labs Diffusion 语言模型系列，自推测模式下吞吐量达
 *          自回归的 6 倍" (fintech-frontier-insights): "三种生成模式" (three
 *          generation modes: 32-token block, iterative denoising, temperature-0
 *          self-speculation equals AR); "训练路线" (training route: block-wise
 *          attention of Efficient-DLM, KV-cache compatibility).
 *   [AIF]  "Nemotron-Labs-Diffusion: 一种统一自回归、扩散和自推测解码的三模式语言
 *          模型" (ai-feeds.com digest): "问题" (AR is causal, diffusion is
 *          bidirectional); "方法 / 推理: 三种模式按需切换" (three inference modes,
 *          one model).
 *   [GSY]  gsyq.cn explainer, §2.3 "自推测解码" (verification rejects the first
 *          mismatching token and everything after it; the target model supplies
 *          the correct token).
 *   [HFB]  "NVIDIA 发布 Nemotron-Labs Diffusion：三模态语言模型统一 AR 与扩散解码"
 *          (aimodeling.com digest of the Hugging Face blog): decode is memory-I/O
 *          bound; fewer refinement steps trade quality for latency.
 *
 * Conventions (all entry points):
 *   - Every call returns an ndiff_status. Argument errors are detected on the
 *     host before anything is enqueued; nothing is launched in that case.
 *   - ndiff_last_error() returns a thread-local, human-readable message for the
 *     last non-OK status returned on the calling thread.
 *   - Device pointers are raw CUDA device addresses owned by the caller; the
 *     library never frees them and never allocates on the kernel entry points.
 *     Work is enqueued asynchronously on the caller's stream (0 = legacy stream).
 *   - Errors found by a kernel are recorded in a device status word and
 *     reported by ndiff_check() (which synchronises the stream): a bounded wait
 *     that expired as NDIFF_ERR_TIMEOUT, a device-side input outside its range
 *     (a kv_len the host cannot see) as NDIFF_ERR_INVALID_ARG.
 *   - The model handle (ndiff_model_*) is the one exception to caller
 *     ownership: it owns its weights, KV cache and scratch.
 */
#ifndef NDIFF_H
#define NDIFF_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define NDIFF_API __attribute__((visibility("default")))
#else
#define NDIFF_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NDIFF_OK = 0,
    NDIFF_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad enum, misaligned */
    NDIFF_ERR_UNSUPPORTED = 2, /* shape/dtype outside the compiled set */
    NDIFF_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
    NDIFF_ERR_OOM = 4,         /* device allocation failed (model handle only) */
    NDIFF_ERR_WORKSPACE = 5,   /* caller workspace smaller than *_workspace_size */
    NDIFF_ERR_TIMEOUT = 6      /* a bounded device-side wait expired */
} ndiff_status;

typedef enum { NDIFF_BF16 = 0, NDIFF_F32 = 1 } ndiff_dtype;

/* Which block keys a block query sees ([TRI] modules; [AIF] "问题"):
 * BIDIR  = every key of the block (diffusion drafting),
 * CAUSAL = block keys up to and including its own slot (AR / verification).
 * Both see the whole committed prefix. */
typedef enum { NDIFF_BIDIR = 0, NDIFF_CAUSAL = 1 } ndiff_mask;

/* The three decode modes of one checkpoint ([FFI] "三种生成模式"). */
typedef enum {
    NDIFF_MODE_AR = 0,
    NDIFF_MODE_DIFF = 1,
    NDIFF_MODE_SELFSPEC = 2,
    NDIFF_MODE_SELFSPEC_FUSED = 3, /* verification of a block and the draft of the next in one forward */
    NDIFF_MODE_SELFSPEC_QUAD = 4   /* verification of a block and drafts of the next for several
                                      acceptance lengths in one forward */
} ndiff_mode;

NDIFF_API const char* ndiff_last_error(void);
NDIFF_API const char* ndiff_status_string(ndiff_status s);

/* Reads back and clears the device status word after synchronising `stream`.
 * Returns NDIFF_ERR_TIMEOUT if any kernel recorded an expired wait since the
 * last check, NDIFF_ERR_INVALID_ARG if a kernel read a device-side input
 * outside its documented range (a kv_len outside [0, Lmax - T], a token id
 * outside [0, vocab)), NDIFF_ERR_CUDA on a CUDA error, else NDIFF_OK. */
NDIFF_API ndiff_status ndiff_check(cudaStream_t stream);

/* Failure-path self-test (a library facility; the pages have no counterpart):
 * enqueues one small kernel whose bounded wait on a barrier that nothing
 * arrives on expires after about limit_us microseconds (1 <= limit_us <=
 * 2000000). The kernel records the expiry in the device status word, the same
 * way every kernel of this library reports an expired wait, and returns; the
 * next ndiff_check() on the stream returns NDIFF_ERR_TIMEOUT and clears the
 * word. Nothing faults and the CUDA context stays usable. */
NDIFF_API ndiff_status ndiff_selftest_timeout(int limit_us, cudaStream_t stream);

/* ------------------------------------------------------------------------ *
 * Block-causal GQA attention over a KV cache ([TRI] modules "Block-wise
 * attention"; [FFI] "三种生成模式": 32-token block; [FFI] "训练路线").
 *
 * For batch b with committed prefix P = kv_len[b], block slot i in [0,T) and
 * query head h (kv head g = h / (Hq/Hkv)):
 *     out[b][i][h] = softmax_j( scale * q[b][i][h] . k[b][g][j] ) . v[b][g][j]
 * over the visible keys j: every j < P, plus the block keys j = P + t with
 * t in [0,T) (BIDIR) or t <= i (CAUSAL). The block's own keys and values must
 * already sit in the cache at positions [P, P+T).
 *
 * Layouts (row-major, contiguous):
 *   q, out            [B][T][Hq][D]
 *   k_cache, v_cache  [B][Hkv][Lmax][D]
 *   kv_len            [B] int32 on the device, 0 <= kv_len[b] <= Lmax - T
 * dt = NDIFF_BF16: bf16 q/k/v/out, fp32 accumulation and softmax; requires
 *   D = 128, (Hq/Hkv) * T <= 128, Hq % Hkv == 0; all pointers 16-byte aligned.
 * dt = NDIFF_F32: fp32 everywhere; requires D <= 64.
 * ws/ws_bytes: device scratch of at least ndiff_block_attn_workspace_size()
 *   bytes (may be NULL when that size is 0). Contents need no initialisation.
 * Values stored in the cache at positions >= kv_len[b] + T are never used
 * (they may hold anything, including NaN). A kv_len outside the range above
 * is an error that only the device sees: the kernels record it in the device
 * status word (the next ndiff_check() returns NDIFF_ERR_INVALID_ARG) and clamp
 * it only to keep every access inside the cache; the output of that call is
 * then meaningless.
 * ------------------------------------------------------------------------ */
NDIFF_API ndiff_status ndiff_block_attn(ndiff_dtype dt, const void* q, const void* k_cache,
                              const void* v_cache, const int32_t* kv_len, int B, int T,
                              int Hq, int Hkv, int D, int Lmax, ndiff_mask mode, float scale,
                              void* out, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Scratch bytes ndiff_block_attn needs for this shape (0 = none). */
NDIFF_API size_t ndiff_block_attn_workspace_size(ndiff_dtype dt, int B, int T, int Hq, int Hkv, int D,
                                       int Lmax);

/* Same as ndiff_block_attn with an explicit KV split length (keys per CTA,
 * a positive multiple of 64; 0 = automatic). The split boundaries sit at
 * absolute key positions, so results for a block row do not depend on T. */
NDIFF_API ndiff_status ndiff_block_attn_split(ndiff_dtype dt, const void* q, const void* k_cache,
                                    const void* v_cache, const int32_t* kv_len, int B, int T,
                                    int Hq, int Hkv, int D, int Lmax, ndiff_mask mode,
                                    float scale, int split_keys, void* out, void* ws,
                                    size_t ws_bytes, cudaStream_t stream);
NDIFF_API size_t ndiff_block_attn_split_workspace_size(ndiff_dtype dt, int B, int T, int Hq, int Hkv,
                                             int D, int Lmax, int split_keys);

/* Same as ndiff_block_attn, for callers that cannot allocate device memory:
 * plugin interfaces that pass a kernel only its inputs and outputs, and
 * processes whose memory manager owns all device memory. The paper has no
 * counterpart; this is a library convenience. The split-KV scratch comes from
 * a static array inside the library of NDIFF_NOALLOC_SCRATCH_BYTES per GPU,
 * held until the process exits; nothing is allocated. Shapes whose
 * ndiff_block_attn_workspace_size() exceeds that size are rejected with
 * NDIFF_ERR_WORKSPACE; argument errors are reported first, as by
 * ndiff_block_attn. The first call on a device looks up the array's device
 * address (again whenever the current CUDA context has changed, e.g. after a
 * cudaDeviceReset) and should come before any stream capture. All calls share the one
 * array: calls whose kernels overlap on the GPU race and must be serialised by
 * the caller. The array keeps what the previous call left in it; nothing in
 * it has to start at zero, because each call writes every partial result
 * before its merge step reads it. */
#define NDIFF_NOALLOC_SCRATCH_BYTES (16u << 20)
NDIFF_API ndiff_status ndiff_block_attn_noalloc(ndiff_dtype dt, const void* q, const void* k_cache,
                                                const void* v_cache, const int32_t* kv_len, int B,
                                                int T, int Hq, int Hkv, int D, int Lmax,
                                                ndiff_mask mode, float scale, void* out,
                                                cudaStream_t stream);

/* ------------------------------------------------------------------------ *
 * Logits reduction: per row r of logits [R][V] (row stride ld elements),
 *   argmax[r] = smallest v in [0,V), v != exclude_id, with the largest logit;
 *               -1 if every id is excluded (V == 1 and exclude_id == 0);
 *   conf[r]   = softmax(row)[argmax[r]] over ALL V ids (the excluded id is in
 *               the normaliser); this is the row's maximum probability unless
 *               the excluded id holds the maximum. 0 when argmax is -1.
 * Greedy (temperature-0) selection is the decision rule of AR decoding and of
 * verification ([FFI] "三种生成模式"); the confidence drives unmasking.
 * dt: NDIFF_BF16 or NDIFF_F32 logits. Logits must be finite.
 * argmax: int32 [R]; conf: float [R] (device). ld >= V; for bf16, ld and the
 * logits pointer must make every row 16-byte aligned (ld % 8 == 0), for f32
 * ld % 4 == 0. R == 0 is a no-op.
 * ------------------------------------------------------------------------ */
NDIFF_API ndiff_status ndiff_logits_reduce(ndiff_dtype dt, const void* logits, int R, int V, int64_t ld,
                                 int exclude_id, int32_t* argmax, float* conf,
                                 cudaStream_t stream);

/* ------------------------------------------------------------------------ *
 * Diffusion unmask step (one denoising round of a block; [FFI]
 * "三种生成模式": iterative denoising of a 32-token block; [HFB]: the number
 * of rounds is the step budget).
 * For each sequence b, among the slots i < T whose bit i of mask_bits[b] is
 * set, select the k' = min(k, popcount) slots of highest conf[b][i] (ties go to
 * the lower slot). For each selected slot i:
 *     draft[b][i] = pred[b][i];  clear bit i of mask_bits[b];
 *     if i <= T-2: block_in[b][i+1] = pred[b][i]   (slot i predicts the token
 *                                                   that input slot i+1 holds)
 * chosen[b][r] = the slot of rank r (r < k'), -1 for r in [k', k).
 * Shapes: conf float [B][T], pred int32 [B][T], mask_bits uint32 [B] (in/out),
 * block_in int32 [B][T] (in/out), draft int32 [B][T] (in/out), chosen int32
 * [B][k]. 1 <= T <= 32, 1 <= k <= T. B == 0 is a no-op. conf must not be NaN.
 * ------------------------------------------------------------------------ */
NDIFF_API ndiff_status ndiff_unmask(const float* conf, const int32_t* pred, int B, int T, int k,
                          uint32_t* mask_bits, int32_t* block_in, int32_t* draft,
                          int32_t* chosen, cudaStream_t stream);

/* ------------------------------------------------------------------------ *
 * Threshold unmask round with revision (the sampler variant of
 * NDIFF_SAMPLER_THRESHOLD; [HFB]: refinement rounds are a budget and earlier
 * tokens can be revised). For each sequence b, with M the masked slots (bits
 * of mask_bits[b]) and E the slots i < T fixed in earlier rounds:
 *   revise: every i in E with pred[b][i] != draft[b][i] and
 *           conf[b][i] >= tau_revise:  draft[b][i] = pred[b][i] and, if
 *           i <= T-2, block_in[b][i+1] = pred[b][i];
 *   fix:    F = { i in M : conf[b][i] >= tau }, or, if F is empty and M is
 *           not, the slot of M with the largest conf (lowest slot on ties);
 *           for i in F: draft[b][i] = pred[b][i], clear bit i, and
 *           block_in[b][i+1] = pred[b][i] if i <= T-2;
 *   n_fixed[b] = |F|, n_revised[b] = revised count (either may be NULL).
 * Comparisons are made on the fp32 values as given. Shapes as in
 * ndiff_unmask; 1 <= T <= 32; tau, tau_revise >= 0 (tau_revise > 1 never
 * revises). B == 0 is a no-op. conf must not be NaN.
 * ------------------------------------------------------------------------ */
NDIFF_API ndiff_status ndiff_unmask_threshold(const float* conf, const int32_t* pred, int B, int T,
                                              float tau, float tau_revise, uint32_t* mask_bits,
                                              int32_t* block_in, int32_t* draft, int32_t* n_fixed,
                                              int32_t* n_revised, cudaStream_t stream);

/* ------------------------------------------------------------------------ *
 * Self-speculation verify / accept ([GSY] §2.3; [FFI] "三种生成模式":
 * diffusion drafts, AR verifies, temperature-0 output equals AR output).
 * For each sequence b:
 *   accept_len[b] = L = first i in [0,T) with draft[b][i] != target[b][i], or T;
 *   n_commit[b]   = n = min(L+1, T)  (the accepted drafts plus the target's
 *                                     correction token when L < T);
 *   commit[b][j]  = target[b][j] for j < n, -1 otherwise;
 *   kv_len[b]    += n   (skipped when kv_len is NULL).
 * Shapes: draft, target, commit int32 [B][T]; accept_len, n_commit, kv_len
 * int32 [B]. 1 <= T <= 32. B == 0 is a no-op.
 * ------------------------------------------------------------------------ */
NDIFF_API ndiff_status ndiff_verify_accept(const int32_t* draft, const int32_t* target, int B, int T,
                                 int32_t* accept_len, int32_t* commit, int32_t* n_commit,
                                 int32_t* kv_len, cudaStream_t stream);

/* ------------------------------------------------------------------------ *
 * Projection of a token block: y[m][n] = sum_k x[m][k] * w[n][k] for m < M,
 * n < N — the matrix products of every layer of the model, which decode runs
 * on at most one 32-token block at a time ([FFI] "三种生成模式"; [HFB]:
 * decode is bound by memory traffic, i.e. by streaming w).
 * x: bf16 [M][K] row-major, w: bf16 [N][K] row-major (both 16-byte aligned),
 * y: fp32 [M][ldy] (ldy >= N). M >= 1, N >= 1, K a positive multiple of 64.
 * fp32 accumulation on the tensor cores. M <= 32 runs the weight-streaming
 * kernel of single-sequence decode (MMA N = 32); larger M, a batch of
 * sequences, runs the wide kernel (MMA N = 256, 256-row token chunks). Within
 * each of the two ranges a row's result does not depend on M (the same row
 * computed alone or inside a larger block is bit-identical).
 * ws/ws_bytes: device scratch of at least ndiff_gemm_bf16_workspace_size()
 *   bytes (0 for M > 32; ws may then be NULL); its contents need no
 *   initialisation (the call clears what it needs).
 * ------------------------------------------------------------------------ */
NDIFF_API size_t ndiff_gemm_bf16_workspace_size(int M, int N, int K);
NDIFF_API ndiff_status ndiff_gemm_bf16(const void* x, const void* w, int M, int N, int K, float* y,
                                       int64_t ldy, void* ws, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------ *
 * LM head with the logits reduction fused in: for token rows m < M,
 *   logits[m][n] = sum_k x[m][k] * w[n][k]   (n < N, never stored)
 *   argmax[m], conf[m] = the reduction of ndiff_logits_reduce over that row
 *   (smallest id of the largest logit with exclude_id left out; its softmax
 *   probability over all N ids).
 * This is the greedy decision of AR decoding and verification, and the
 * confidence of the unmask step, taken straight from the last hidden state
 * ([FFI] "三种生成模式"; [HFB]: decode is bound by memory traffic, and this
 * removes the write and re-read of the [M][N] logits).
 * x: bf16 [M][K] row-major, w: bf16 [N][K] row-major (16-byte aligned);
 * M >= 1 (M > 32: the wide kernel, as in ndiff_gemm_bf16), N >= 1, K a
 * positive multiple of 64, -1 <= exclude_id < N.
 * argmax int32 [M], conf float [M] (device). The logits are the fp32 values
 * ndiff_gemm_bf16 produces, so argmax equals ndiff_gemm_bf16 followed by
 * ndiff_logits_reduce exactly; conf agrees to fp32 rounding. A row's results
 * do not depend on M within M <= 32, nor within M > 32.
 * ws/ws_bytes: device scratch of at least ndiff_lm_head_argmax_workspace_size()
 *   bytes; contents need no initialisation.
 * ------------------------------------------------------------------------ */
NDIFF_API size_t ndiff_lm_head_argmax_workspace_size(int M, int N, int K);
NDIFF_API ndiff_status ndiff_lm_head_argmax(const void* x, const void* w, int M, int N, int K,
                                            int exclude_id, int32_t* argmax, float* conf, void* ws,
                                            size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------ *
 * Random-init tri-mode model (one checkpoint, three modes: [FFI]
 * "三种生成模式"; [AIF] "方法 / 推理").
 * Pre-norm transformer: x = E[ids]; per layer
 *   h = RMSNorm(x); q,k,v = h Wq^T, h Wk^T, h Wv^T; RoPE(q,k);
 *   x += BlockAttn(q,k,v) Wo^T; h = RMSNorm(x); x += (silu(h Wg^T) * h Wu^T) Wd^T;
 * logits = RMSNorm(x) Wlm^T. RMSNorm gain 1, eps cfg.eps, RoPE rotate-half with
 * base cfg.rope_base. Every weight ~ N(0, 0.02^2) drawn with Philox4x64-10
 * (Salmon et al., SC'11) and Box-Muller from `seed`: element i of tensor t
 * takes the output words (w0..w3) of counter (i/4, t, 0, 0) under key
 * (seed, 0); lanes i%4 = 0/1 use (w0, w1), lanes 2/3 use (w2, w3), with
 * u1 = ((wa >> 11) + 1) 2^-53, u2 = (wb >> 11) 2^-53, z = sqrt(-2 ln u1) times
 * cos (even lane) or sin (odd lane) of 2 pi u2; the weight is float(0.02 z),
 * then bf16 (round to nearest even) for bf16 models. Tensor ids: 0 embedding,
 * 1 + 8 l + j for layer l (j = 0 q, 1 k, 2 v, 3 o, 4 gate, 5 up, 6 down),
 * 1 + 8 layers the LM head. The [MASK] id is vocab-1 and is never predicted.
 * dtype NDIFF_F32: fp32 weights/activations (tiny configs: d_model <= 1024,
 *   head_dim <= 64, vocab <= 65536).
 * dtype NDIFF_BF16: bf16 weights, bf16 GEMM inputs, fp32 residual stream and
 *   accumulators; requires head_dim == 128, d_model % 128 == 0, ffn % 128 == 0,
 *   n_heads/n_kv_heads * 32 <= 128.
 * batch: sequences decoded together. 1 serves the single-sequence calls
 *   (ndiff_prefill, ndiff_decode_step[_ex], ndiff_model_forward); B > 1 (bf16
 *   models only) serves the batch calls (ndiff_prefill_batch,
 *   ndiff_decode_step_batch), which run every projection on the wide kernel
 *   over B*T token rows and attention over B ragged sequences ([TRI] Abstract:
 *   the modes serve different deployment settings and concurrency levels).
 * ------------------------------------------------------------------------ */
typedef struct {
    int layers;
    int d_model;
    int n_heads;
    int n_kv_heads;
    int head_dim;
    int ffn;
    int vocab;
    ndiff_dtype dtype;
    float rope_base;
    float eps;
    int max_seq; /* KV cache capacity in tokens (prompt + generated + 32) */
    int batch;   /* sequences decoded together (1 .. 4096; > 1 needs bf16) */
} ndiff_model_config;

typedef struct ndiff_model ndiff_model;

typedef struct {
    int64_t forwards;        /* model forwards run by the calls so far (prefill excluded) */
    int64_t tokens;          /* tokens committed by the calls so far */
    int32_t last_accept_len; /* L of the last SELFSPEC verification (-1 otherwise) */
    int32_t last_n_commit;   /* tokens committed by the last decode step */
    int64_t accept_hist[33]; /* histogram of L over SELFSPEC verifications */
    int64_t revisions;       /* earlier draft tokens replaced (threshold sampler) */
    int32_t last_rounds;     /* drafting forwards of the last decode step */
    int32_t reserved;
} ndiff_stats;

/* How a DIFF or SELFSPEC block is drafted ([FFI] "三种生成模式": a block is
 * denoised over several rounds; [HFB]: the number of rounds is a budget the
 * user sets, and the model can revise tokens it already produced; [AIF]
 * 核心洞察: the sampler decides how many tokens a forward yields).
 *   NDIFF_SAMPLER_TOPK:      `steps` rounds, each fixing the k = 32/steps most
 *                            confident masked slots (ndiff_unmask).
 *   NDIFF_SAMPLER_THRESHOLD: rounds until no slot is masked (at most 32), each
 *                            fixing every masked slot with confidence >= tau
 *                            or else the most confident one, after replacing
 *                            earlier slots' tokens whose new prediction differs
 *                            with confidence >= tau_revise (> 1: no revision)
 *                            (ndiff_unmask_threshold). */
typedef enum { NDIFF_SAMPLER_TOPK = 0, NDIFF_SAMPLER_THRESHOLD = 1 } ndiff_sampler;

typedef struct {
    ndiff_mode mode;
    ndiff_sampler sampler;
    int steps;          /* TOPK: 1 <= steps <= 32, 32 % steps == 0 */
    float tau;          /* THRESHOLD: fix threshold, 0 <= tau */
    float tau_revise;   /* THRESHOLD: revision threshold, 0 <= tau_revise (> 1: off) */
    int n_cand;         /* SELFSPEC_QUAD: candidate acceptance lengths besides 32 (1 or 2) */
    int cand[2];        /* SELFSPEC_QUAD: the candidates, each in [0, 32) */
} ndiff_decode_opts;

NDIFF_API ndiff_status ndiff_model_create(const ndiff_model_config* cfg, uint64_t seed, ndiff_model** out);
NDIFF_API ndiff_status ndiff_model_destroy(ndiff_model* m);

/* Causal forward over prompt[0..n-2] (host ids) that fills the KV cache;
 * prompt[n-1] becomes the pending "last" token. Resets the session.
 * 1 <= n, n + 32 <= max_seq. Synchronous on return. */
NDIFF_API ndiff_status ndiff_prefill(ndiff_model* m, const int32_t* prompt_host, int n,
                           cudaStream_t stream);

/* One decode cycle in `mode` (shifted convention: the logits of input slot i
 * predict the token after it):
 *   AR:       one forward of [last] (CAUSAL); commits 1 token.
 *   DIFF:     `steps` forwards of the 32-slot block [last, MASK x 31]
 *             (BIDIR), each unmasking k = 32/steps slots, then one BIDIR
 *             forward of the finished block that writes its KV; commits 32
 *             tokens.
 *   SELFSPEC: the DIFF draft (steps forwards) then one CAUSAL forward of
 *             [last, d0..d30]; commits the accepted prefix plus the correction.
 *   SELFSPEC_FUSED (bf16, one sequence): unless the previous cycle left a
 *             draft of this block, one BIDIR drafting forward; then one
 *             forward of 64 rows that verifies [last, d0..d30] (CAUSAL) and
 *             drafts the next block [d31, MASK x 31] at the following 32
 *             positions (BIDIR over the prefix and the verified block, as if
 *             it is accepted whole). Commits the accepted prefix plus the
 *             correction; when all 32 drafts were accepted, the second half's
 *             argmaxes are the next cycle's draft ([FFI] 吞吐量数据: linear
 *             self-speculation). Needs max_seq >= committed + 64.
 *   SELFSPEC_QUAD (bf16, one sequence; ndiff_decode_step_ex with n_cand and
 *             cand, ndiff_decode_step uses the candidates 0 and 1): as
 *             SELFSPEC_FUSED, and the same forward also drafts the next block
 *             for each candidate acceptance length L < 32: 32 [MASK] inputs
 *             at positions P+L+1 .. P+L+32 (BIDIR) over the prefix plus the
 *             verified block's first L+1 inputs (the state after committing L
 *             drafts and the correction, whose slot stays masked because the
 *             forward cannot know it). When the verified L is 32 or a
 *             candidate, that block's argmaxes are the next cycle's draft
 *             ([FFI] 吞吐量数据: quadratic self-speculation). 128 rows per
 *             forward; needs max_seq >= committed + 448 (the candidate blocks'
 *             K/V sit in cache rows past the verified block).
 * steps: drafting forwards per block (1 <= steps <= 32, 32 % steps == 0);
 *   ignored for AR and SELFSPEC_FUSED (one drafting forward).
 * out_tokens_host: host buffer of >= 32 int32; *n_out receives the count.
 * stats (optional) accumulates counters. Synchronous on return. */
NDIFF_API ndiff_status ndiff_decode_step(ndiff_model* m, ndiff_mode mode, int steps,
                               int32_t* out_tokens_host, int* n_out, ndiff_stats* stats,
                               cudaStream_t stream);

/* ndiff_decode_step with a choice of draft sampler (see ndiff_decode_opts) and,
 * for NDIFF_MODE_SELFSPEC_QUAD, of the candidate acceptance lengths.
 * With NDIFF_SAMPLER_THRESHOLD the rounds run one after another with a 4-byte
 * read of the block's mask word between them (the round count depends on the
 * model's confidence); every round and the final forward are CUDA graphs.
 * AR ignores the sampler. Synchronous on return. */
NDIFF_API ndiff_status ndiff_decode_step_ex(ndiff_model* m, const ndiff_decode_opts* opts,
                                            int32_t* out_tokens_host, int* n_out,
                                            ndiff_stats* stats, cudaStream_t stream);

/* Batched sessions (cfg.batch = B > 1). Prefill: prompt b is
 * prompts_host[sum_{c<b} lengths_host[c] ..] of lengths_host[b] tokens
 * (1 <= n_b, n_b + 32 <= max_seq); each sequence's cache takes its prompt but
 * the last token, which becomes its pending token. The prompts advance 32
 * tokens per forward together; a sequence whose prompt is used up runs filler
 * tokens past its prefix (scratch cache rows that the next block overwrites).
 * Synchronous on return. */
NDIFF_API ndiff_status ndiff_prefill_batch(ndiff_model* m, const int32_t* prompts_host,
                                           const int32_t* lengths_host, cudaStream_t stream);

/* One decode cycle of all B sequences in opts->mode (as ndiff_decode_step_ex):
 * every forward runs the B blocks (or B pending tokens in AR) together, and
 * unmasking, verification and commits are per sequence, so accept lengths
 * differ from sequence to sequence. out_tokens_host [B][32] receives sequence
 * b's committed tokens in row b, n_out_host [B] their counts. stats counts
 * batch forwards and the tokens of all sequences; accept_hist counts every
 * sequence's verification. The fixed-schedule cycle is one CUDA graph.
 * Synchronous on return. */
NDIFF_API ndiff_status ndiff_decode_step_batch(ndiff_model* m, const ndiff_decode_opts* opts,
                                               int32_t* out_tokens_host, int32_t* n_out_host,
                                               ndiff_stats* stats, cudaStream_t stream);

/* Per-sequence committed prefix lengths and pending tokens ([B] host arrays,
 * either may be NULL). */
NDIFF_API ndiff_status ndiff_model_state_batch(const ndiff_model* m, int32_t* kv_len_host,
                                               int32_t* last_host);

/* Runs one forward of `T` block tokens (host ids) at the model's current
 * position with the given mask, writes fp32 logits [T][vocab] to the host
 * buffer (may be NULL) and returns them without changing the session (the
 * block's KV entries beyond the committed prefix are scratch). For parity
 * tests and diagnostics. Synchronous. */
NDIFF_API ndiff_status ndiff_model_forward(ndiff_model* m, const int32_t* ids_host, int T,
                                 ndiff_mask mode, float* logits_host, cudaStream_t stream);

/* Session state readout: committed prefix length (KV entries) and the pending
 * last token. */
NDIFF_API ndiff_status ndiff_model_state(const ndiff_model* m, int* kv_len, int32_t* last_token);

/* Copies `count` elements of weight tensor `tensor_id` starting at flat
 * element `offset` (the Philox element index of that tensor) to the host as
 * fp32. For tests of the weight generator. Synchronous. */
NDIFF_API ndiff_status ndiff_model_read_weight(const ndiff_model* m, int tensor_id, int64_t offset,
                                     int64_t count, float* host_out);

#ifdef __cplusplus
}
#endif

#endif /* NDIFF_H */
