// model.cu — the random-init tri-mode model behind the C ABI: weights, KV
// caches, one forward of a token block, and the decode modes (AR, block
// diffusion, self-speculation with top-k or threshold drafts, fused
// verify + draft self-speculation), for one sequence or a batch of ragged
// sequences decoded together.
//
// Sources (page title, section):
//   "NVIDIA 发布 Nemotron-Labs Diffusion 语言模型系列" (fintech-frontier-insights),
//     "三种生成模式": one checkpoint run as AR (token by token), as block
//     diffusion (a 32-token block refined over several denoising rounds) or as
//     self-speculation (diffusion drafts, AR verifies; at temperature 0 the
//     output equals AR output); "训练路线": block-wise attention keeps the KV
//     cache usable.
//   "Nemotron-Labs-Diffusion: A Tri-Mode Language Model ..." (hotpaper.ai),
//     Abstract: in self-speculation the diffusion mode drafts and the AR mode
//     verifies, within one model.
//   gsyq.cn explainer, §2.3 "自推测解码": accept the agreeing prefix and take
//     the verifier's token at the first mismatch.
//
// Readings where the pages are silent: the logits of input slot i predict the
// token after it in every mode; [MASK] = vocab-1, never predicted; a diffusion
// block enters the cache through one bidirectional forward of the finished
// block; the self-speculation draft is `steps` bidirectional forwards, each
// fixing the 32/steps most confident masked slots (or, with the threshold
// sampler, every masked slot at or above tau, with revision of earlier slots);
// the fused mode verifies a block and drafts the next one in a 64-row forward.
//
// Numerics: bf16 models keep bf16 weights and round the inputs of every matrix
// product (normed activations, attention output, SwiGLU output) and q/k/v to
// bf16; the residual stream, accumulators and logits are fp32. Every kernel
// computes a token row independently of the other rows and of the block
// length, so a causal block forward reproduces single-token forwards bit for
// bit and temperature-0 self-speculation commits exactly the AR tokens.
#include <math.h>
#include <string.h>

#include <functional>
#include <map>
#include <tuple>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "model_kernels.h"

using namespace ndiff;

#define TRY(expr)                                 \
  do {                                            \
    ndiff_status _s = (expr);                     \
    if (_s != NDIFF_OK) return _s;                \
  } while (0)

namespace {

constexpr int kBlock = 32;
constexpr double kSigma = 0.02;

struct Layer {
  void* wqkv = nullptr;  // [(Hq + 2 Hkv) D][d]: q rows, k rows, v rows
  void* wo = nullptr;    // [d][Hq D]
  void* wgu = nullptr;   // [2 ffn][d]: bf16 64-row interleave of gate/up; f32 gate then up
  void* wd = nullptr;    // [d][ffn]
  void* kc = nullptr;    // [Hkv][Lmax][D]
  void* vc = nullptr;
  CUtensorMap tm_qkv, tm_o, tm_gu, tm_d;
};

}  // namespace

struct ndiff_model {
  ndiff_model_config cfg;
  uint64_t seed = 0;
  int dev = 0;
  bool bf16 = false;
  size_t esz = 4;
  int D = 0, Hq = 0, Hkv = 0, d = 0, ffn = 0, V = 0, L = 0, Lmax = 0, NQKV = 0, HD = 0;
  int32_t mask_id = 0;
  float eps = 1e-6f;
  void* embed = nullptr;
  void* lm = nullptr;
  std::vector<Layer> layers;
  // activations (32 token rows)
  float* x = nullptr;        // residual stream fp32 [32][d]
  void* h = nullptr;         // normed input [32][d] (bf16 or f32)
  void* qb = nullptr;        // q [32][Hq][D]
  void* ob = nullptr;        // attention output [32][Hq D]
  void* ab = nullptr;        // SwiGLU output [32][ffn]
  float* y = nullptr;        // fp32 path projection scratch [32][ymax]
  int B = 1;                 // sequences decoded together; activations hold B * 32 rows
  float* logits = nullptr;   // [32][ldl] fp32 (rows 16-byte aligned)
  int ldl = 0;
  // decode-cycle state
  int32_t* ids = nullptr;       // [32] forward input of AR / model_forward
  int32_t* pred = nullptr;      // [32] argmax
  float* conf = nullptr;        // [32]
  int32_t* draft = nullptr;     // [32]
  int32_t* block_in = nullptr;  // [32]
  // per-sequence results, one contiguous block for the host read:
  // commit [B][32] | n_commit [B] | accept_len [B] | fixed [B] | revised [B]
  int32_t* res = nullptr;
  int32_t* commit = nullptr;
  int32_t* ncommit = nullptr;
  int32_t* acclen = nullptr;
  int32_t* nfixed = nullptr;
  int32_t* nrevised = nullptr;
  int32_t* kv_len = nullptr;    // [B]
  uint32_t* mask = nullptr;     // [B]
  int32_t* chosen = nullptr;    // [32]
  int32_t* prompt = nullptr;    // [Lmax]
  float2* rope = nullptr;       // [Lmax][D/2]
  float* gws = nullptr;         // GEMM split partials
  float4* red = nullptr;        // LM head per-tile argmax partials [tiles][32]
  int* gcnt = nullptr;          // GEMM tile counters
  void* aws = nullptr;          // attention split-KV scratch
  size_t aws_bytes = 0;
  int attn_split = 0;
  int attn_split_quad = 0;      // the quadratic forward's three draft blocks (one launch)
  CUtensorMap tm_h, tm_oact, tm_a, tm_lm;
  CUtensorMap tm_h_w, tm_oact_w, tm_a_w;  // 256-row boxes for the wide kernel (B > 1)
  CUtensorMap tm_h_w64, tm_oact_w64, tm_a_w64;  // 64-row boxes: its AR forwards (B <= 64 rows)
  CUtensorMap tm_h64, tm_oact64, tm_a64;  // 64-row boxes: the fused verify + draft forward
  CUtensorMap tm_h128, tm_oact128, tm_a128;  // 128-row boxes: the quadratic forward
  int32_t* fin = nullptr;       // [128] fused / quadratic forward input
  int32_t* kv_len2 = nullptr;   // [1] prefix of the fused forward's draft half
  int32_t* kvc = nullptr;       // [4] quadratic forward: prefixes of its three draft blocks
  int4* remap = nullptr;        // [4] quadratic forward: their key remaps
  int32_t* blk_pos = nullptr;   // [8] quadratic forward: position and cache row of each block
  int32_t* cand_dev = nullptr;  // [2] candidate acceptance lengths of the quadratic mode
  int cand_host[2] = {-1, -1};
  bool have_draft = false;      // the last fused forward left a draft of the next block
  int last_L0 = -1;             // accept length of sequence 0 in the last verification
  GemmPlan pl_qkv, pl_o, pl_gu, pl_d, pl_lm;
  int32_t* pin = nullptr;       // pinned host staging [pin_n]
  size_t pin_n = 0;
  int32_t* last_dev = nullptr;  // [B] pending last token per sequence
  cudaStream_t ms = nullptr;    // the model's own stream (decode graphs run here)
  // decode graphs by (part, mode, steps, tau bits, tau_revise bits)
  std::map<std::tuple<int, int, int, uint32_t, uint32_t>, cudaGraphExec_t> graphs;
  std::vector<void*> allocs;
  std::vector<int> P;          // committed prefix per sequence (host view)
  std::vector<int32_t> last;   // pending token per sequence (host view)
  bool ready = false;
};

namespace {

ndiff_status dalloc(ndiff_model* m, void** p, size_t bytes) {
  *p = nullptr;
  cudaError_t e = cudaMalloc(p, bytes ? bytes : 16);
  if (e != cudaSuccess) {
    cudaGetLastError();
    *p = nullptr;
    return set_error(NDIFF_ERR_OOM, "ndiff_model_create: cudaMalloc of %zu bytes failed (%s)", bytes,
                     cudaGetErrorString(e));
  }
  m->allocs.push_back(*p);
  return NDIFF_OK;
}

template <typename Tp>
ndiff_status dalloc_t(ndiff_model* m, Tp** p, size_t bytes) {
  void* v = nullptr;
  ndiff_status s = dalloc(m, &v, bytes);
  *p = static_cast<Tp*>(v);
  return s;
}

void free_model(ndiff_model* m) {
  for (auto& kv : m->graphs) cudaGraphExecDestroy(kv.second);
  m->graphs.clear();
  if (m->ms) cudaStreamDestroy(m->ms);
  m->ms = nullptr;
  for (void* p : m->allocs) cudaFree(p);
  m->allocs.clear();
  if (m->pin) cudaFreeHost(m->pin);
  m->pin = nullptr;
}

int tid_layer(int l, int j) { return 1 + 8 * l + j; }

ndiff_status check_config(const ndiff_model_config* c) {
  if (!c) return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_model_create: null config");
  if (c->layers < 1 || c->d_model < 1 || c->n_heads < 1 || c->n_kv_heads < 1 || c->head_dim < 2 ||
      c->ffn < 1 || c->vocab < 2 || c->max_seq < kBlock + 1 || !(c->eps > 0.f) ||
      !(c->rope_base > 1.f))
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_model_create: bad sizes in config");
  if (c->batch < 1 || c->batch > 4096)
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_model_create: batch in [1, 4096] (got %d)", c->batch);
  if (c->batch > 1 && c->dtype != NDIFF_BF16)
    return set_error(NDIFF_ERR_UNSUPPORTED, "ndiff_model_create: batch > 1 needs a bf16 model");
  if (c->n_heads % c->n_kv_heads != 0 || c->head_dim % 2 != 0)
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_model_create: n_heads %% n_kv_heads and head_dim %% 2 must be 0");
  if (c->dtype == NDIFF_BF16) {
    if (c->head_dim != 128 || c->d_model % 128 != 0 || c->ffn % 128 != 0 ||
        (c->n_heads / c->n_kv_heads) * kBlock > 128)
      return set_error(NDIFF_ERR_UNSUPPORTED,
                       "ndiff_model_create: bf16 models need head_dim 128, d_model and ffn multiples "
                       "of 128, and n_heads/n_kv_heads <= 4");
    if ((long long)c->batch * c->n_kv_heads * c->max_seq >= (1LL << 31))
      return set_error(NDIFF_ERR_UNSUPPORTED, "ndiff_model_create: KV cache too large");
  } else if (c->dtype == NDIFF_F32) {
    if (c->head_dim > 64 || c->d_model > 4096 || c->vocab > (1 << 20))
      return set_error(NDIFF_ERR_UNSUPPORTED,
                       "ndiff_model_create: fp32 models need head_dim <= 64, d_model <= 4096");
  } else {
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_model_create: bad dtype %d", (int)c->dtype);
  }
  return NDIFF_OK;
}

// ---------------------------------------------------------------- one forward
// What a forward leaves behind: nothing (the KV cache only), the argmax /
// confidence of every row in m->pred / m->conf, or those plus the fp32 logits
// in m->logits. For bf16 models FWD_TOKENS never stores logits: the LM head
// GEMM reduces each 128-id vocabulary tile in its epilogue and a merge kernel
// folds the tiles.
enum { FWD_NONE = 0, FWD_TOKENS = 1, FWD_LOGITS = 2 };

// Runs T (<= 32) tokens of each of the B sequences (`ids` [B][T], device) at
// positions kv_len[b] .. kv_len[b]+T-1 and writes their K/V into each
// sequence's cache there. A single sequence uses the weight-streaming kernel
// (MMA N = 32); a batch uses the wide kernel (MMA N = 256) for every
// projection, so a row's arithmetic is the same in AR (T = 1) and block
// (T = 32) forwards either way.
//
// T = 64 (one bf16 sequence) is the fused forward of two blocks: rows 0..31
// are a block under verification (CAUSAL at prefix kv_len) and rows 32..63 the
// next block to draft (BIDIR at prefix kv_len + 32, read from kv_len2); the
// projections run the 64-column kernel, whose per-row arithmetic is that of
// the 32-column one.
ndiff_status forward(ndiff_model* m, const int32_t* ids, int T, int causal, int out,
                     cudaStream_t s) {
  PdlScope pdl(m->bf16);
  const float scale = 1.f / sqrtf((float)m->D);
  const int B = m->B, M = B * T;
  const bool wide = B > 1;
  const bool fused = T == 2 * kBlock;
  const bool quad = T == 4 * kBlock;
  if ((fused || quad) && (wide || !m->bf16))
    return set_error(NDIFF_ERR_UNSUPPORTED, "fused verify + draft forward: one bf16 sequence only");
  const int mt = quad ? 4 * kBlock : (fused ? 2 * kBlock : kBlock);
  TRY(launch_embed(m->embed, m->bf16, ids, M, m->V, m->d, m->x, s));
  GemmParams gp;
  memset(&gp, 0, sizeof(gp));
  gp.T = M;
  gp.Tb = T;
  gp.w_tiled = 1;
  gp.ws = m->gws;
  gp.counters = m->gcnt;
  // one projection: W [N][K] against the activation behind tx (skinny) / txw (wide)
  // the activation maps of one projection input: 32-row boxes (one block),
  // 64-row boxes (fused forward), and the wide kernel's 256- and 64-row boxes
  struct XMaps {
    const CUtensorMap &x32, &x64, &x128, &w256, &w64;
  };
  const XMaps xh{m->tm_h, m->tm_h64, m->tm_h128, m->tm_h_w, m->tm_h_w64};
  const XMaps xo{m->tm_oact, m->tm_oact64, m->tm_oact128, m->tm_oact_w, m->tm_oact_w64};
  const XMaps xa{m->tm_a, m->tm_a64, m->tm_a128, m->tm_a_w, m->tm_a_w64};
  auto proj = [&](const CUtensorMap& tw, const XMaps& xm, const GemmPlan& pl, int N, int K,
                  const GemmParams& p) -> ndiff_status {
    if (wide)
      return launch_gemm_wide(tw, gemm_wide_box_rows(M) == 64 ? xm.w64 : xm.w256,
                              gemm_wide_plan(N, K, M), p, s);
    if (fused) return launch_gemm_bf16(tw, xm.x64, pl, p, s, mt);
    if (quad) return launch_gemm_bf16(tw, xm.x128, pl, p, s, mt);
    return launch_gemm_bf16(tw, xm.x32, pl, p, s);
  };
  // One bf16 sequence: every layer projection leaves its partial tiles unsummed
  // (GEMM_EPI_PARTIAL, no merge at the projection's end) and the kernel after
  // it sums them: the QKV merge (RoPE, q and the block's K/V), the residual
  // add fused with the next RMSNorm (output and down projections), the SwiGLU
  // merge. A batch runs the wide kernel with its fused epilogues.
  const bool defer = m->bf16 && !wide;
  auto pp_of = [&](const GemmPlan& pl) {
    PartialPlan pp;
    pp.part = m->gws;
    pp.nks = pl.nks;
    pp.U = pl.ntiles * pl.nks;
    pp.G = pl.grid;
    pp.maxseg = gemm_plan_maxseg(pl);
    return pp;
  };
  auto norm_after = [&](bool partial, const GemmPlan& pl) -> ndiff_status {
    if (!partial) return launch_rmsnorm(m->x, M, m->d, m->eps, m->h, m->bf16, s);
    return launch_residual_rmsnorm(m->x, M, m->d, m->eps, static_cast<__nv_bfloat16*>(m->h), pp_of(pl),
                                   mt, s);
  };
  for (int l = 0; l < m->L; ++l) {
    Layer& ly = m->layers[l];
    TRY(norm_after(l > 0 && defer, m->pl_d));
    if (m->bf16) {
      GemmParams p = gp;
      p.N = m->NQKV;
      p.mode = defer ? GEMM_EPI_PARTIAL : GEMM_EPI_QKV;
      p.maxseg = gemm_plan_maxseg(m->pl_qkv);
      p.q = static_cast<__nv_bfloat16*>(m->qb);
      p.kc = static_cast<__nv_bfloat16*>(ly.kc);
      p.vc = static_cast<__nv_bfloat16*>(ly.vc);
      p.Hq = m->Hq;
      p.Hkv = m->Hkv;
      p.Lmax = m->Lmax;
      p.kv_len = m->kv_len;
      p.rope = m->rope;
      p.blk_pos = quad ? m->blk_pos : nullptr;
      TRY(proj(ly.tm_qkv, xh, m->pl_qkv, m->NQKV, m->d, p));
      if (defer)
        TRY(launch_qkv_merge(pp_of(m->pl_qkv), M, m->Hq, m->Hkv, m->Lmax, m->kv_len, p.blk_pos, m->rope,
                             p.q, p.kc, p.vc, mt, s));
      if (quad) {
        // the block under verification (causal at prefix P), then its three
        // draft blocks as one batch over the same cache (bidirectional, each at
        // its own prefix, the candidate blocks' keys remapped to their rows)
        const size_t blk = (size_t)kBlock * m->HD;
        __nv_bfloat16* qb = static_cast<__nv_bfloat16*>(m->qb);
        __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(m->ob);
        TRY(launch_attn_bf16(qb, ly.kc, ly.vc, m->kv_len, 1, kBlock, m->Hq, m->Hkv, m->Lmax, 1,
                             scale, m->attn_split, ob, m->aws, m->aws_bytes, s, nullptr, 0, 1));
        TRY(launch_attn_bf16(qb + blk, ly.kc, ly.vc, m->kvc, 3, kBlock, m->Hq, m->Hkv, m->Lmax, 0,
                             scale, m->attn_split_quad, ob + blk, m->aws, m->aws_bytes, s, m->remap,
                             1));
      } else if (fused) {
        const size_t half = (size_t)kBlock * m->HD;  // elements of one block's q / output rows
        __nv_bfloat16* qb = static_cast<__nv_bfloat16*>(m->qb);
        __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(m->ob);
        TRY(launch_attn_bf16(qb, ly.kc, ly.vc, m->kv_len, 1, kBlock, m->Hq, m->Hkv, m->Lmax, 1,
                             scale, m->attn_split, ob, m->aws, m->aws_bytes, s, nullptr, 0, 1, ly.wo,
                             (size_t)m->d * m->HD * 2));
        TRY(launch_attn_bf16(qb + half, ly.kc, ly.vc, m->kv_len2, 1, kBlock, m->Hq, m->Hkv,
                             m->Lmax, 0, scale, m->attn_split, ob + half, m->aws, m->aws_bytes, s));
      } else {
        // one sequence: the QKV merge before it lets the prefix K/V stream early,
        // and the attention CTAs pull the output projection's weights into L2
        // while HBM would otherwise idle; a block's longer attention also pulls
        // the gate/up projection's next six k-steps of every run
        const bool blk_pf = defer && T >= kBlock;
        TRY(launch_attn_bf16(m->qb, ly.kc, ly.vc, m->kv_len, B, T, m->Hq, m->Hkv, m->Lmax, causal,
                             scale, m->attn_split, m->ob, m->aws, m->aws_bytes, s, nullptr, 0,
                             defer ? 1 : 0, defer ? ly.wo : nullptr,
                             defer ? (size_t)m->d * m->HD * 2 : 0, blk_pf ? ly.wgu : nullptr,
                             m->pl_gu.ntiles * m->pl_gu.nks, m->pl_gu.grid));
      }
      p = gp;
      p.N = m->d;
      p.mode = defer ? GEMM_EPI_PARTIAL : GEMM_EPI_RESID;
      p.maxseg = gemm_plan_maxseg(m->pl_o);
      p.out = m->x;
      p.ldo = m->d;
      TRY(proj(ly.tm_o, xo, m->pl_o, m->d, m->HD, p));
      TRY(norm_after(defer, m->pl_o));
      p = gp;
      p.N = 2 * m->ffn;
      p.mode = defer ? GEMM_EPI_PARTIAL : GEMM_EPI_SWIGLU;
      p.maxseg = gemm_plan_maxseg(m->pl_gu);
      p.act = static_cast<__nv_bfloat16*>(m->ab);
      p.lda = m->ffn;
      TRY(proj(ly.tm_gu, xh, m->pl_gu, 2 * m->ffn, m->d, p));
      if (defer)
        TRY(launch_swiglu_merge(pp_of(m->pl_gu), m->pl_gu.ntiles, M, p.act, p.lda, mt, s));
      p = gp;
      p.N = m->d;
      p.mode = defer ? GEMM_EPI_PARTIAL : GEMM_EPI_RESID;
      p.maxseg = gemm_plan_maxseg(m->pl_d);
      p.out = m->x;
      p.ldo = m->d;
      TRY(proj(ly.tm_d, xa, m->pl_d, m->d, m->ffn, p));
    } else {
      const float* h = static_cast<const float*>(m->h);
      TRY(launch_linear_f32(h, m->d, static_cast<const float*>(ly.wqkv), m->NQKV, m->d, m->y,
                            m->NQKV, T, s));
      TRY(launch_qkv_rope_f32(m->y, T, m->Hq, m->Hkv, m->D, m->Lmax, m->kv_len, m->rope,
                              static_cast<float*>(m->qb), static_cast<float*>(ly.kc),
                              static_cast<float*>(ly.vc), s));
      TRY(launch_attn_f32(static_cast<const float*>(m->qb), static_cast<const float*>(ly.kc),
                          static_cast<const float*>(ly.vc), m->kv_len, 1, T, m->Hq, m->Hkv, m->D,
                          m->Lmax, causal, scale, static_cast<float*>(m->ob), s));
      TRY(launch_linear_f32(static_cast<const float*>(m->ob), m->HD, static_cast<const float*>(ly.wo),
                            m->d, m->HD, m->y, m->d, T, s));
      TRY(launch_resid_add_f32(m->x, m->y, T * m->d, s));
      TRY(launch_rmsnorm(m->x, T, m->d, m->eps, m->h, false, s));
      TRY(launch_linear_f32(h, m->d, static_cast<const float*>(ly.wgu), 2 * m->ffn, m->d, m->y,
                            2 * m->ffn, T, s));
      TRY(launch_swiglu_f32(m->y, T, m->ffn, static_cast<float*>(m->ab), s));
      TRY(launch_linear_f32(static_cast<const float*>(m->ab), m->ffn, static_cast<const float*>(ly.wd),
                            m->d, m->ffn, m->y, m->d, T, s));
      TRY(launch_resid_add_f32(m->x, m->y, T * m->d, s));
    }
  }
  // (a forward that leaves nothing but the KV cache needs no final residual)
  if (out == FWD_NONE) return NDIFF_OK;
  TRY(norm_after(defer, m->pl_d));
  if (m->bf16 && out == FWD_TOKENS) {
    GemmParams p = gp;
    p.N = m->V;
    p.mode = GEMM_EPI_ARGMAX;
    p.red = m->red;
    p.excl = m->mask_id;
    TRY(proj(m->tm_lm, xh, m->pl_lm, m->V, m->d, p));
    return launch_argmax_merge(m->red, m->pl_lm.ntiles, M, wide ? M : mt, m->pred, m->conf, s);
  }
  if (wide || fused || quad)
    return set_error(NDIFF_ERR_UNSUPPORTED, "model logits: one block of one sequence only");
  if (m->bf16) {
    GemmParams p = gp;
    p.N = m->V;
    p.mode = GEMM_EPI_F32;
    p.out = m->logits;
    p.ldo = m->ldl;
    TRY(launch_gemm_bf16(m->tm_lm, m->tm_h, m->pl_lm, p, s));
  } else {
    TRY(launch_linear_f32(static_cast<const float*>(m->h), m->d, static_cast<const float*>(m->lm),
                          m->V, m->d, m->logits, m->ldl, T, s));
  }
  return launch_logits_reduce(NDIFF_F32, m->logits, T, m->V, m->ldl, m->mask_id, m->pred, m->conf, s);
}

// Fills the 32-slot draft of the next block: `steps` bidirectional forwards,
// each fixing the k = 32/steps most confident masked slots.
ndiff_status draft_block(ndiff_model* m, int steps, cudaStream_t s) {
  const int k = kBlock / steps;
  TRY(launch_block_init(m->block_in, m->draft, m->mask, kBlock, m->last_dev, m->mask_id, m->B, s));
  for (int i = 0; i < steps; ++i) {
    TRY(forward(m, m->block_in, kBlock, 0, FWD_TOKENS, s));
    TRY(launch_unmask(m->conf, m->pred, m->B, kBlock, k, m->mask, m->block_in, m->draft, m->chosen,
                      s));
  }
  return NDIFF_OK;
}

// The end of a DIFF or SELFSPEC cycle, once the draft is complete.
ndiff_status enqueue_tail(ndiff_model* m, ndiff_mode mode, cudaStream_t s) {
  if (mode == NDIFF_MODE_DIFF) {
    // the finished block enters the cache through one bidirectional forward
    TRY(forward(m, m->block_in, kBlock, 0, FWD_NONE, s));
    return launch_commit(m->draft, kBlock, nullptr, kBlock, kBlock, m->last_dev, m->kv_len, m->B, s);
  }
  // SELFSPEC: causal verification of [last, d0..d30], accept the agreeing prefix
  TRY(forward(m, m->block_in, kBlock, 1, FWD_TOKENS, s));
  TRY(launch_verify_accept(m->draft, m->pred, m->B, kBlock, m->acclen, m->commit, m->ncommit,
                           m->kv_len, s));
  return launch_commit(m->commit, kBlock, m->ncommit, 0, 0, m->last_dev, m->kv_len, m->B, s);
}

// Enqueues one decode cycle; every input it reads (pending token, committed
// prefix) lives on the device, so the same launches can be replayed.
ndiff_status enqueue_cycle(ndiff_model* m, ndiff_mode mode, int steps, cudaStream_t s) {
  if (mode == NDIFF_MODE_AR) {
    // AR: one causal forward of [last]; commit its argmax.
    TRY(forward(m, m->last_dev, 1, 1, FWD_TOKENS, s));
    return launch_commit(m->pred, 1, nullptr, 1, 1, m->last_dev, m->kv_len, m->B, s);
  }
  TRY(draft_block(m, steps, s));
  return enqueue_tail(m, mode, s);
}

// One cycle of fused self-speculation (one sequence): unless the previous
// fused forward left a draft of this block, a drafting forward first; then one
// forward verifies the block (rows 0..31, CAUSAL) and drafts the next
// (rows 32..63, BIDIR, as if the whole block is accepted); the agreeing
// prefix plus the correction is committed, and when all 32 drafts were
// accepted the draft half becomes the next block's draft.
ndiff_status enqueue_fused(ndiff_model* m, bool need_draft, cudaStream_t s) {
  if (need_draft) TRY(draft_block(m, 1, s));
  TRY(launch_fused_input(m->fin, m->block_in, m->draft, m->mask_id, m->kv_len, m->kv_len2, s));
  TRY(forward(m, m->fin, 2 * kBlock, 1, FWD_TOKENS, s));
  TRY(launch_verify_accept(m->draft, m->pred, 1, kBlock, m->acclen, m->commit, m->ncommit,
                           m->kv_len, s));
  TRY(launch_commit(m->commit, kBlock, m->ncommit, 0, 0, m->last_dev, m->kv_len, 1, s));
  return launch_fused_stash(m->pred + kBlock, m->acclen, m->last_dev, m->draft, m->block_in, s);
}

// One cycle of quadratic self-speculation (one sequence): as enqueue_fused,
// with one forward of 128 rows that verifies the block and drafts the next
// for full acceptance and for the two candidate acceptance lengths in
// m->cand_dev; the draft of the verified length, if drafted, is stashed.
ndiff_status enqueue_quad(ndiff_model* m, bool need_draft, cudaStream_t s) {
  if (need_draft) TRY(draft_block(m, 1, s));
  TRY(launch_quad_input(m->fin, m->block_in, m->draft, m->mask_id, m->kv_len, m->cand_dev, m->kvc,
                        m->remap, m->blk_pos, s));
  TRY(forward(m, m->fin, 4 * kBlock, 1, FWD_TOKENS, s));
  TRY(launch_verify_accept(m->draft, m->pred, 1, kBlock, m->acclen, m->commit, m->ncommit,
                           m->kv_len, s));
  TRY(launch_commit(m->commit, kBlock, m->ncommit, 0, 0, m->last_dev, m->kv_len, 1, s));
  return launch_quad_stash(m->pred, m->acclen, m->cand_dev, m->last_dev, m->draft, m->block_in, s);
}

enum { PART_CYCLE = 0, PART_INIT = 1, PART_ROUND = 2, PART_TAIL = 3, PART_FUSED = 4, PART_QUAD = 5 };

// The launches `fn` enqueues, as an instantiated CUDA graph captured on the
// model's stream on first use and kept under `key`.
ndiff_status cached_graph(ndiff_model* m, const std::tuple<int, int, int, uint32_t, uint32_t>& key,
                          const std::function<ndiff_status(cudaStream_t)>& fn,
                          cudaGraphExec_t* out) {
  auto it = m->graphs.find(key);
  if (it != m->graphs.end()) {
    *out = it->second;
    return NDIFF_OK;
  }
  NDIFF_CUDA_TRY(cudaStreamBeginCapture(m->ms, cudaStreamCaptureModeThreadLocal));
  ndiff_status st = fn(m->ms);
  cudaGraph_t g = nullptr;
  cudaError_t e = cudaStreamEndCapture(m->ms, &g);
  if (st != NDIFF_OK) {
    if (g) cudaGraphDestroy(g);
    return st;
  }
  if (e != cudaSuccess) return cuda_error(e, "cudaStreamEndCapture");
  cudaGraphExec_t ge = nullptr;
  e = cudaGraphInstantiate(&ge, g, 0);
  cudaGraphDestroy(g);
  if (e != cudaSuccess) return cuda_error(e, "cudaGraphInstantiate");
  m->graphs[key] = ge;
  *out = ge;
  return NDIFF_OK;
}

// The decode cycle of a fixed schedule (AR, or a top-k draft of `steps` rounds).
ndiff_status cycle_graph(ndiff_model* m, ndiff_mode mode, int steps, cudaGraphExec_t* out) {
  const int st = mode == NDIFF_MODE_AR ? 0 : steps;
  return cached_graph(m, std::make_tuple((int)PART_CYCLE, (int)mode, st, 0u, 0u),
                      [&](cudaStream_t s) { return enqueue_cycle(m, mode, steps, s); }, out);
}

// Waits for the stream and reports device-side timeouts recorded meanwhile.
ndiff_status finish(cudaStream_t s) {
  NDIFF_CUDA_TRY(cudaStreamSynchronize(s));
  unsigned int* w = device_status_word();
  if (w) {
    unsigned int v = 0;
    NDIFF_CUDA_TRY(cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost));
    if (v) {
      unsigned int z = 0;
      NDIFF_CUDA_TRY(cudaMemcpy(w, &z, sizeof(z), cudaMemcpyHostToDevice));
      if (v & kStatusTimeout)
        return set_error(NDIFF_ERR_TIMEOUT, "a bounded device wait expired (status 0x%x)", v);
      return set_error(NDIFF_ERR_INVALID_ARG,
                       "a kernel read an input outside its range (status 0x%x)", v);
    }
  }
  return NDIFF_OK;
}

ndiff_status set_device(const ndiff_model* m) {
  int cur = -1;
  NDIFF_CUDA_TRY(cudaGetDevice(&cur));
  if (cur != m->dev) NDIFF_CUDA_TRY(cudaSetDevice(m->dev));
  return NDIFF_OK;
}

ndiff_status create(const ndiff_model_config* cfg, uint64_t seed, ndiff_model* m) {
  const ndiff_model_config& c = *cfg;
  m->cfg = c;
  m->seed = seed;
  NDIFF_CUDA_TRY(cudaGetDevice(&m->dev));
  m->bf16 = c.dtype == NDIFF_BF16;
  m->esz = m->bf16 ? 2 : 4;
  m->D = c.head_dim;
  m->Hq = c.n_heads;
  m->Hkv = c.n_kv_heads;
  m->d = c.d_model;
  m->ffn = c.ffn;
  m->V = c.vocab;
  m->L = c.layers;
  m->Lmax = c.max_seq;
  m->HD = m->Hq * m->D;
  m->NQKV = (m->Hq + 2 * m->Hkv) * m->D;
  m->mask_id = m->V - 1;
  m->ldl = (m->V + 3) & ~3;
  m->eps = c.eps;
  m->B = c.batch;
  m->P.assign(m->B, 0);
  m->last.assign(m->B, -1);
  const size_t esz = m->esz;
  const size_t d = m->d;
  // activation rows: B blocks, or the four blocks of a quadratic forward
  const size_t R = (size_t)(m->B > 1 ? m->B * kBlock : 4 * kBlock);
  cudaStream_t s = 0;

  TRY(dalloc(m, &m->embed, (size_t)m->V * d * esz));
  const size_t vpad = (size_t)((m->V + 127) / 128) * 128;  // whole 128-row tiles
  TRY(dalloc(m, &m->lm, vpad * d * esz));
  NDIFF_CUDA_TRY(cudaMemsetAsync(m->lm, 0, vpad * d * esz, s));
  m->layers.resize(m->L);
  const size_t kv_elems = (size_t)m->B * m->Hkv * m->Lmax * m->D;
  for (Layer& ly : m->layers) {
    TRY(dalloc(m, &ly.wqkv, (size_t)m->NQKV * d * esz));
    TRY(dalloc(m, &ly.wo, d * m->HD * esz));
    TRY(dalloc(m, &ly.wgu, 2 * (size_t)m->ffn * d * esz));
    TRY(dalloc(m, &ly.wd, d * m->ffn * esz));
    TRY(dalloc(m, &ly.kc, kv_elems * esz));
    TRY(dalloc(m, &ly.vc, kv_elems * esz));
    NDIFF_CUDA_TRY(cudaMemsetAsync(ly.kc, 0, kv_elems * esz, s));
    NDIFF_CUDA_TRY(cudaMemsetAsync(ly.vc, 0, kv_elems * esz, s));
  }
  const int ymax = m->NQKV > 2 * m->ffn ? m->NQKV : 2 * m->ffn;
  TRY(dalloc_t(m, &m->x, R * d * 4));
  TRY(dalloc(m, &m->h, R * d * esz));
  TRY(dalloc(m, &m->qb, R * m->HD * esz));
  TRY(dalloc(m, &m->ob, R * m->HD * esz));
  TRY(dalloc(m, &m->ab, R * m->ffn * esz));
  TRY(dalloc_t(m, &m->y, (size_t)kBlock * (ymax > m->d ? ymax : m->d) * 4));
  TRY(dalloc_t(m, &m->logits, (size_t)kBlock * m->ldl * 4));
  NDIFF_CUDA_TRY(cudaMemsetAsync(m->x, 0, R * d * 4, s));
  NDIFF_CUDA_TRY(cudaMemsetAsync(m->h, 0, R * d * esz, s));
  NDIFF_CUDA_TRY(cudaMemsetAsync(m->qb, 0, R * m->HD * esz, s));
  NDIFF_CUDA_TRY(cudaMemsetAsync(m->ob, 0, R * m->HD * esz, s));
  NDIFF_CUDA_TRY(cudaMemsetAsync(m->ab, 0, R * m->ffn * esz, s));
  TRY(dalloc_t(m, &m->ids, R * 4));
  TRY(dalloc_t(m, &m->pred, R * 4));
  TRY(dalloc_t(m, &m->conf, R * 4));
  TRY(dalloc_t(m, &m->draft, R * 4));
  TRY(dalloc_t(m, &m->block_in, R * 4));
  const size_t Bn = (size_t)m->B;
  const size_t RC = Bn * kBlock;  // commit rows
  TRY(dalloc_t(m, &m->res, (RC + 4 * Bn) * 4));
  m->commit = m->res;
  m->ncommit = m->res + RC;
  m->acclen = m->ncommit + Bn;
  m->nfixed = m->acclen + Bn;
  m->nrevised = m->nfixed + Bn;
  TRY(dalloc_t(m, &m->kv_len, Bn * 4));
  TRY(dalloc_t(m, &m->mask, Bn * 4));
  TRY(dalloc_t(m, &m->chosen, R * 4));
  TRY(dalloc_t(m, &m->prompt, (size_t)m->Lmax * 4));
  TRY(dalloc_t(m, &m->last_dev, Bn * 4));
  TRY(dalloc_t(m, &m->fin, 4 * kBlock * 4));
  TRY(dalloc_t(m, &m->kvc, 16));
  TRY(dalloc_t(m, &m->remap, 4 * sizeof(int4)));
  TRY(dalloc_t(m, &m->blk_pos, 8 * 4));
  TRY(dalloc_t(m, &m->cand_dev, 16));
  NDIFF_CUDA_TRY(cudaMemsetAsync(m->remap, 0, 4 * sizeof(int4), s));
  NDIFF_CUDA_TRY(cudaMemsetAsync(m->cand_dev, 0, 16, s));
  TRY(dalloc_t(m, &m->kv_len2, 16));
  TRY(dalloc_t(m, &m->rope, (size_t)m->Lmax * (m->D / 2) * sizeof(float2)));
  NDIFF_CUDA_TRY(cudaMemsetAsync(m->ids, 0, R * 4, s));
  NDIFF_CUDA_TRY(cudaMemsetAsync(m->kv_len, 0, Bn * 4, s));
  NDIFF_CUDA_TRY(cudaMemsetAsync(m->last_dev, 0, Bn * 4, s));
  NDIFF_CUDA_TRY(cudaMemsetAsync(m->block_in, 0, R * 4, s));

  if (m->bf16) {
    m->pl_qkv = gemm_plan(m->NQKV, m->d);
    m->pl_o = gemm_plan(m->d, m->HD);
    m->pl_gu = gemm_plan(2 * m->ffn, m->d);
    m->pl_d = gemm_plan(m->d, m->ffn);
    m->pl_lm = gemm_plan(m->V, m->d);

    const GemmPlan* pls[5] = {&m->pl_qkv, &m->pl_o, &m->pl_gu, &m->pl_d, &m->pl_lm};
    size_t ws = 16;
    int tiles = 1;
    const int mtmax = m->B > 1 ? 2 * kBlock : 4 * kBlock;
    for (const GemmPlan* pl : pls) {
      size_t b = gemm_partials_bytes(*pl, mtmax);
      if (pl != &m->pl_lm && m->B == 1) {  // the layer projections leave unsummed partials
        const size_t b2 = gemm_partial_only_bytes(*pl, mtmax);
        b = b2 > b ? b2 : b;
      }
      if (b > ws) ws = b;
      if (pl->ntiles > tiles) tiles = pl->ntiles;
    }
    TRY(dalloc_t(m, &m->gws, ws));
    TRY(dalloc_t(m, &m->gcnt, (size_t)tiles * 4));
    TRY(dalloc_t(m, &m->red, (size_t)m->pl_lm.ntiles * R * sizeof(float4)));
    NDIFF_CUDA_TRY(cudaMemsetAsync(m->gcnt, 0, (size_t)tiles * 4, s));
    m->attn_split = attn_bf16_auto_split(m->B, m->Hkv, m->Lmax);
    m->aws_bytes = attn_bf16_workspace(m->B, kBlock, m->Hq, m->Hkv, m->Lmax, m->attn_split);
    if (m->B == 1) {
      // The quadratic forward's three draft blocks run as one batch with a split
      // length of their own (the block under verification keeps the AR split:
      // its rows must match single-token forwards bit for bit; draft rows need not).
      m->attn_split_quad = attn_bf16_auto_split(3, m->Hkv, m->Lmax);
      const size_t q3 = attn_bf16_workspace(3, kBlock, m->Hq, m->Hkv, m->Lmax, m->attn_split_quad);
      if (q3 > m->aws_bytes) m->aws_bytes = q3;
    }
    if (m->aws_bytes) TRY(dalloc(m, &m->aws, m->aws_bytes));
    TRY(gemm_make_maps(nullptr, 0, m->d, false, m->h, kBlock, nullptr, &m->tm_h));
    TRY(gemm_make_maps(nullptr, 0, m->HD, false, m->ob, kBlock, nullptr, &m->tm_oact));
    TRY(gemm_make_maps(nullptr, 0, m->ffn, false, m->ab, kBlock, nullptr, &m->tm_a));
    TRY(gemm_make_maps(nullptr, 0, m->d, false, m->h, 2 * kBlock, nullptr, &m->tm_h64, 2 * kBlock));
    TRY(gemm_make_maps(nullptr, 0, m->HD, false, m->ob, 2 * kBlock, nullptr, &m->tm_oact64,
                       2 * kBlock));
    TRY(gemm_make_maps(nullptr, 0, m->ffn, false, m->ab, 2 * kBlock, nullptr, &m->tm_a64,
                       2 * kBlock));
    if (m->B == 1) {
      TRY(gemm_make_maps(nullptr, 0, m->d, false, m->h, 4 * kBlock, nullptr, &m->tm_h128, 4 * kBlock));
      TRY(gemm_make_maps(nullptr, 0, m->HD, false, m->ob, 4 * kBlock, nullptr, &m->tm_oact128,
                         4 * kBlock));
      TRY(gemm_make_maps(nullptr, 0, m->ffn, false, m->ab, 4 * kBlock, nullptr, &m->tm_a128,
                         4 * kBlock));
    }
    TRY(gemm_wide_make_xmap(m->h, (int)R, m->d, &m->tm_h_w));
    TRY(gemm_wide_make_xmap(m->ob, (int)R, m->HD, &m->tm_oact_w));
    TRY(gemm_wide_make_xmap(m->ab, (int)R, m->ffn, &m->tm_a_w));
    TRY(gemm_wide_make_xmap(m->h, (int)R, m->d, &m->tm_h_w64, 64));
    TRY(gemm_wide_make_xmap(m->ob, (int)R, m->HD, &m->tm_oact_w64, 64));
    TRY(gemm_wide_make_xmap(m->ab, (int)R, m->ffn, &m->tm_a_w64, 64));
    TRY(gemm_make_maps(m->lm, m->V, m->d, true, nullptr, 0, &m->tm_lm, nullptr));
    for (Layer& ly : m->layers) {
      TRY(gemm_make_maps(ly.wqkv, m->NQKV, m->d, true, nullptr, 0, &ly.tm_qkv, nullptr));
      TRY(gemm_make_maps(ly.wo, m->d, m->HD, true, nullptr, 0, &ly.tm_o, nullptr));
      TRY(gemm_make_maps(ly.wgu, 2 * m->ffn, m->d, true, nullptr, 0, &ly.tm_gu, nullptr));
      TRY(gemm_make_maps(ly.wd, m->d, m->ffn, true, nullptr, 0, &ly.tm_d, nullptr));
    }
  }

  // weights: tensor ids 0 = embedding, 1 + 8 l + j for layer l
  // (j: 0 q, 1 k, 2 v, 3 o, 4 gate, 5 up, 6 down), 1 + 8 L = LM head
  const bool b = m->bf16;
  // bf16 projection weights are stored as contiguous 128 x 64 tiles (each TMA
  // box of the projection kernel is then one 16 KB run of HBM); the embedding
  // is read by rows and stays row-major.
  TRY(launch_init_normal(m->embed, b, 0, m->V, m->d, 0, ROWMAP_IDENTITY, false, seed, kSigma, s));
  for (int l = 0; l < m->L; ++l) {
    Layer& ly = m->layers[l];
    const int64_t kvr = (int64_t)m->Hkv * m->D;
    const int qk_map = b ? ROWMAP_ROPE : ROWMAP_IDENTITY;
    TRY(launch_init_normal(ly.wqkv, b, tid_layer(l, 0), m->HD, m->d, 0, qk_map, b, seed, kSigma, s));
    TRY(launch_init_normal(ly.wqkv, b, tid_layer(l, 1), kvr, m->d, m->HD, qk_map, b, seed, kSigma, s));
    TRY(launch_init_normal(ly.wqkv, b, tid_layer(l, 2), kvr, m->d, m->HD + kvr, ROWMAP_IDENTITY, b, seed,
                           kSigma, s));
    TRY(launch_init_normal(ly.wo, b, tid_layer(l, 3), m->d, m->HD, 0, ROWMAP_IDENTITY, b, seed, kSigma, s));
    TRY(launch_init_normal(ly.wgu, b, tid_layer(l, 4), m->ffn, m->d, 0, b ? ROWMAP_GATE : ROWMAP_IDENTITY,
                           b, seed, kSigma, s));
    TRY(launch_init_normal(ly.wgu, b, tid_layer(l, 5), m->ffn, m->d, b ? 0 : m->ffn,
                           b ? ROWMAP_UP : ROWMAP_IDENTITY, b, seed, kSigma, s));
    TRY(launch_init_normal(ly.wd, b, tid_layer(l, 6), m->d, m->ffn, 0, ROWMAP_IDENTITY, b, seed, kSigma, s));
  }
  TRY(launch_init_normal(m->lm, b, 1 + 8 * m->L, m->V, m->d, 0, ROWMAP_IDENTITY, b, seed, kSigma, s));
  TRY(launch_rope_table(m->rope, m->Lmax, m->D, (double)c.rope_base, s));

  // host staging: the largest read (SELFSPEC results, R + 2 B ints), a
  // threshold round's masks and counts (3 B), a prefill chunk (R + B)
  m->pin_n = R + 8 * Bn + 64;
  cudaError_t e = cudaMallocHost(reinterpret_cast<void**>(&m->pin), m->pin_n * sizeof(int32_t));
  if (e != cudaSuccess) {
    m->pin = nullptr;
    return set_error(NDIFF_ERR_OOM, "ndiff_model_create: pinned host buffer: %s", cudaGetErrorString(e));
  }
  NDIFF_CUDA_TRY(cudaStreamCreateWithFlags(&m->ms, cudaStreamNonBlocking));
  NDIFF_CUDA_TRY(cudaStreamSynchronize(s));
  // One forward of each block length sets every kernel attribute and device
  // lookup up front, so that later graph captures only record launches. The
  // cache rows it writes are scratch until a prefill fills them.
  TRY(forward(m, m->ids, 1, 1, m->B > 1 ? FWD_TOKENS : FWD_LOGITS, m->ms));
  TRY(forward(m, m->block_in, kBlock, 0, FWD_TOKENS, m->ms));
  TRY(finish(m->ms));
  NDIFF_CUDA_TRY(cudaGetLastError());
  return NDIFF_OK;
}

// Locates weight tensor `tid`: storage base, columns, first storage row, row map.
bool locate(const ndiff_model* m, int tid, const void** base, int64_t* rows, int64_t* cols,
            int64_t* row_off, int* map, bool* tiled) {
  *row_off = 0;
  *map = ROWMAP_IDENTITY;
  *tiled = m->bf16 && tid != 0;
  if (tid == 0 || tid == 1 + 8 * m->L) {
    *base = tid == 0 ? m->embed : m->lm;
    *rows = m->V;
    *cols = m->d;
    return true;
  }
  if (tid < 1 || tid > 8 * m->L) return false;
  const int l = (tid - 1) / 8, j = (tid - 1) % 8;
  const Layer& ly = m->layers[l];
  const int64_t kvr = (int64_t)m->Hkv * m->D;
  switch (j) {
    case 0:
      *base = ly.wqkv; *rows = m->HD; *cols = m->d;
      if (m->bf16) *map = ROWMAP_ROPE;
      return true;
    case 1:
      *base = ly.wqkv; *rows = kvr; *cols = m->d; *row_off = m->HD;
      if (m->bf16) *map = ROWMAP_ROPE;
      return true;
    case 2: *base = ly.wqkv; *rows = kvr; *cols = m->d; *row_off = m->HD + kvr; return true;
    case 3: *base = ly.wo; *rows = m->d; *cols = m->HD; return true;
    case 4:
      *base = ly.wgu; *rows = m->ffn; *cols = m->d;
      if (m->bf16) *map = ROWMAP_GATE;
      return true;
    case 5:
      *base = ly.wgu; *rows = m->ffn; *cols = m->d;
      if (m->bf16) *map = ROWMAP_UP; else *row_off = m->ffn;
      return true;
    case 6: *base = ly.wd; *rows = m->d; *cols = m->ffn; return true;
    default: return false;
  }
}

}  // namespace

extern "C" {

ndiff_status ndiff_model_create(const ndiff_model_config* cfg, uint64_t seed, ndiff_model** out) {
  if (!out) return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_model_create: null output pointer");
  *out = nullptr;
  TRY(check_config(cfg));
  ndiff_model* m = new ndiff_model();
  ndiff_status st = create(cfg, seed, m);
  if (st != NDIFF_OK) {
    free_model(m);
    delete m;
    return st;
  }
  *out = m;
  return NDIFF_OK;
}

ndiff_status ndiff_model_destroy(ndiff_model* m) {
  if (!m) return NDIFF_OK;
  set_device(m);
  cudaDeviceSynchronize();
  free_model(m);
  delete m;
  return NDIFF_OK;
}

ndiff_status ndiff_prefill(ndiff_model* m, const int32_t* prompt_host, int n, cudaStream_t stream) {
  if (!m || !prompt_host) return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_prefill: null pointer");
  if (m->B != 1)
    return set_error(NDIFF_ERR_UNSUPPORTED, "ndiff_prefill: batched model; use ndiff_prefill_batch");
  if (n < 1 || n + kBlock > m->Lmax)
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_prefill: need 1 <= n and n + 32 <= max_seq (n=%d, max_seq=%d)",
                     n, m->Lmax);
  for (int i = 0; i < n; ++i)
    if (prompt_host[i] < 0 || prompt_host[i] >= m->V)
      return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_prefill: token %d at %d out of range", prompt_host[i], i);
  TRY(set_device(m));
  m->ready = false;
  m->have_draft = false;
  NDIFF_CUDA_TRY(cudaMemsetAsync(m->kv_len, 0, sizeof(int32_t), stream));
  NDIFF_CUDA_TRY(cudaMemcpyAsync(m->prompt, prompt_host, (size_t)n * 4, cudaMemcpyHostToDevice, stream));
  for (int off = 0; off < n - 1; off += kBlock) {
    const int T = (n - 1 - off) < kBlock ? (n - 1 - off) : kBlock;
    TRY(forward(m, m->prompt + off, T, 1, FWD_NONE, stream));
    TRY(launch_kv_add(m->kv_len, T, stream));
  }
  m->pin[0] = prompt_host[n - 1];
  NDIFF_CUDA_TRY(cudaMemcpyAsync(m->last_dev, m->pin, 4, cudaMemcpyHostToDevice, stream));
  TRY(finish(stream));
  m->P[0] = n - 1;
  m->last[0] = prompt_host[n - 1];
  m->ready = true;
  return NDIFF_OK;
}

ndiff_status ndiff_prefill_batch(ndiff_model* m, const int32_t* prompts_host,
                                 const int32_t* lengths_host, cudaStream_t stream) {
  if (!m || !prompts_host || !lengths_host)
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_prefill_batch: null pointer");
  const int B = m->B;
  std::vector<int64_t> off(B + 1, 0);
  int longest = 0;
  for (int b = 0; b < B; ++b) {
    const int n = lengths_host[b];
    if (n < 1 || n + kBlock > m->Lmax)
      return set_error(NDIFF_ERR_INVALID_ARG,
                       "ndiff_prefill_batch: sequence %d: need 1 <= n and n + 32 <= max_seq (n=%d)", b, n);
    off[b + 1] = off[b] + n;
    longest = n > longest ? n : longest;
  }
  for (int64_t i = 0; i < off[B]; ++i)
    if (prompts_host[i] < 0 || prompts_host[i] >= m->V)
      return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_prefill_batch: token out of range at %lld",
                       (long long)i);
  TRY(set_device(m));
  m->ready = false;
  m->have_draft = false;
  // All sequences advance through their prompts 32 tokens per forward. A
  // sequence whose prompt is used up runs filler tokens at positions past its
  // prefix; those cache rows are scratch (the next block overwrites them) and
  // no committed row attends to them.
  const size_t R = (size_t)B * kBlock;
  int32_t* ids = m->pin;
  int32_t* kv = m->pin + R;
  for (int c = 0; c * kBlock < longest - 1; ++c) {
    for (int b = 0; b < B; ++b) {
      const int n1 = lengths_host[b] - 1;  // prompt[0 .. n-2] enters the cache
      const int p0 = c * kBlock < n1 ? c * kBlock : n1;
      kv[b] = p0;
      for (int i = 0; i < kBlock; ++i)
        ids[(size_t)b * kBlock + i] = (p0 + i < n1 && c * kBlock + i < n1)
                                          ? prompts_host[off[b] + c * kBlock + i]
                                          : 0;
    }
    NDIFF_CUDA_TRY(cudaMemcpyAsync(m->ids, ids, R * 4, cudaMemcpyHostToDevice, stream));
    NDIFF_CUDA_TRY(cudaMemcpyAsync(m->kv_len, kv, (size_t)B * 4, cudaMemcpyHostToDevice, stream));
    TRY(forward(m, m->ids, kBlock, 1, FWD_NONE, stream));
    TRY(finish(stream));  // the staging buffer is rewritten for the next chunk
  }
  for (int b = 0; b < B; ++b) {
    kv[b] = lengths_host[b] - 1;
    ids[b] = prompts_host[off[b + 1] - 1];
  }
  NDIFF_CUDA_TRY(cudaMemcpyAsync(m->kv_len, kv, (size_t)B * 4, cudaMemcpyHostToDevice, stream));
  NDIFF_CUDA_TRY(cudaMemcpyAsync(m->last_dev, ids, (size_t)B * 4, cudaMemcpyHostToDevice, stream));
  TRY(finish(stream));
  for (int b = 0; b < B; ++b) {
    m->P[b] = lengths_host[b] - 1;
    m->last[b] = prompts_host[off[b + 1] - 1];
  }
  m->ready = true;
  return NDIFF_OK;
}

// Reads the committed tokens of the cycle just enqueued on the model's stream
// (out_tokens_host [B][32], n_out [B]) and advances the host view of each
// session.
static ndiff_status collect(ndiff_model* m, ndiff_mode mode, int64_t forwards, int rounds,
                            int64_t revisions, int32_t* out_tokens_host, int32_t* n_out,
                            ndiff_stats* stats) {
  const int B = m->B;
  const size_t R = (size_t)B * kBlock;
  if (mode == NDIFF_MODE_AR)
    NDIFF_CUDA_TRY(cudaMemcpyAsync(m->pin, m->pred, (size_t)B * 4, cudaMemcpyDeviceToHost, m->ms));
  else if (mode == NDIFF_MODE_DIFF)
    NDIFF_CUDA_TRY(cudaMemcpyAsync(m->pin, m->draft, R * 4, cudaMemcpyDeviceToHost, m->ms));
  else
    NDIFF_CUDA_TRY(cudaMemcpyAsync(m->pin, m->res, (R + 2 * B) * 4, cudaMemcpyDeviceToHost, m->ms));
  TRY(finish(m->ms));
  int64_t tokens = 0;
  for (int b = 0; b < B; ++b) {
    int n = 0, L = -1;
    const int32_t* src = nullptr;
    if (mode == NDIFF_MODE_AR) {
      n = 1;
      src = m->pin + b;
    } else if (mode == NDIFF_MODE_DIFF) {
      n = kBlock;
      src = m->pin + (size_t)b * kBlock;
    } else {
      n = m->pin[R + b];
      L = m->pin[R + B + b];
      src = m->pin + (size_t)b * kBlock;
    }
    for (int i = 0; i < n; ++i) out_tokens_host[(size_t)b * kBlock + i] = src[i];
    n_out[b] = n;
    if (b == 0) m->last_L0 = L;
    m->P[b] += n;
    m->last[b] = src[n - 1];
    tokens += n;
    if (stats) {
      if (b == 0) {
        stats->last_accept_len = L;
        stats->last_n_commit = n;
      }
      if (L >= 0 && L <= kBlock) stats->accept_hist[L] += 1;
    }
  }
  if (stats) {
    stats->forwards += forwards;
    stats->tokens += tokens;
    stats->revisions += revisions;
    stats->last_rounds = rounds;
  }
  return NDIFF_OK;
}

// One decode cycle of every sequence of the model (see ndiff_decode_step_ex).
static ndiff_status decode_cycle(ndiff_model* m, const ndiff_decode_opts* opts,
                                 int32_t* out_tokens_host, int32_t* n_out, ndiff_stats* stats,
                                 cudaStream_t stream) {
  const ndiff_mode mode = opts->mode;
  if (!m->ready) return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_decode_step: no prefill yet");
  if (mode != NDIFF_MODE_AR && mode != NDIFF_MODE_DIFF && mode != NDIFF_MODE_SELFSPEC &&
      mode != NDIFF_MODE_SELFSPEC_FUSED && mode != NDIFF_MODE_SELFSPEC_QUAD)
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_decode_step: bad mode %d", (int)mode);
  if (mode == NDIFF_MODE_SELFSPEC_QUAD) {
    if (m->B != 1 || !m->bf16)
      return set_error(NDIFF_ERR_UNSUPPORTED,
                       "ndiff_decode_step: quadratic self-speculation needs one bf16 sequence");
    if (opts->n_cand < 1 || opts->n_cand > 2)
      return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_decode_step: n_cand must be 1 or 2 (got %d)",
                       opts->n_cand);
    const int c0 = opts->cand[0], c1 = opts->n_cand > 1 ? opts->cand[1] : opts->cand[0];
    if (c0 < 0 || c0 >= kBlock || c1 < 0 || c1 >= kBlock)
      return set_error(NDIFF_ERR_INVALID_ARG,
                       "ndiff_decode_step: candidate acceptance lengths must be in [0, 32) (got %d, %d)",
                       c0, c1);
    if (m->P[0] + 448 > m->Lmax)
      return set_error(NDIFF_ERR_INVALID_ARG,
                       "ndiff_decode_step: quadratic mode needs max_seq >= committed + 448 (%d of %d)",
                       m->P[0], m->Lmax);
    TRY(set_device(m));
    NDIFF_CUDA_TRY(cudaStreamSynchronize(stream));
    if (c0 != m->cand_host[0] || c1 != m->cand_host[1]) {
      const int32_t hc[2] = {c0, c1};
      NDIFF_CUDA_TRY(cudaMemcpy(m->cand_dev, hc, sizeof(hc), cudaMemcpyHostToDevice));
      m->cand_host[0] = c0;
      m->cand_host[1] = c1;
    }
    const bool need = !m->have_draft;
    cudaGraphExec_t ge = nullptr;
    TRY(cached_graph(m, std::make_tuple((int)PART_QUAD, (int)mode, need ? 1 : 0, 0u, 0u),
                     [&](cudaStream_t s2) { return enqueue_quad(m, need, s2); }, &ge));
    NDIFF_CUDA_TRY(cudaGraphLaunch(ge, m->ms));
    TRY(collect(m, mode, need ? 2 : 1, need ? 1 : 0, 0, out_tokens_host, n_out, stats));
    m->have_draft = m->last_L0 == kBlock || m->last_L0 == c0 || m->last_L0 == c1;
    return NDIFF_OK;
  }
  if (mode == NDIFF_MODE_SELFSPEC_FUSED) {
    if (m->B != 1 || !m->bf16)
      return set_error(NDIFF_ERR_UNSUPPORTED,
                       "ndiff_decode_step: fused self-speculation needs one bf16 sequence");
    for (int b = 0; b < m->B; ++b)
      if (m->P[b] + 2 * kBlock > m->Lmax)
        return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_decode_step: KV cache full (%d of %d)",
                         m->P[b], m->Lmax);
    TRY(set_device(m));
    NDIFF_CUDA_TRY(cudaStreamSynchronize(stream));
    const bool need = !m->have_draft;
    cudaGraphExec_t ge = nullptr;
    TRY(cached_graph(m, std::make_tuple((int)PART_FUSED, (int)mode, need ? 1 : 0, 0u, 0u),
                     [&](cudaStream_t s2) { return enqueue_fused(m, need, s2); }, &ge));
    NDIFF_CUDA_TRY(cudaGraphLaunch(ge, m->ms));
    TRY(collect(m, mode, need ? 2 : 1, need ? 1 : 0, 0, out_tokens_host, n_out, stats));
    m->have_draft = m->last_L0 == kBlock;
    return NDIFF_OK;
  }
  const bool thr = mode != NDIFF_MODE_AR && opts->sampler == NDIFF_SAMPLER_THRESHOLD;
  if (mode != NDIFF_MODE_AR) {
    if (opts->sampler != NDIFF_SAMPLER_TOPK && opts->sampler != NDIFF_SAMPLER_THRESHOLD)
      return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_decode_step: bad sampler %d", (int)opts->sampler);
    if (!thr && (opts->steps < 1 || opts->steps > kBlock || kBlock % opts->steps != 0))
      return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_decode_step: steps must divide 32 (got %d)",
                       opts->steps);
    if (thr && !(opts->tau >= 0.f && opts->tau_revise >= 0.f))
      return set_error(NDIFF_ERR_INVALID_ARG,
                       "ndiff_decode_step: tau and tau_revise must be >= 0 (got %g, %g)",
                       (double)opts->tau, (double)opts->tau_revise);
  }
  const int need = mode == NDIFF_MODE_AR ? 1 : kBlock;
  for (int b = 0; b < m->B; ++b)
    if (m->P[b] + need > m->Lmax)
      return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_decode_step: KV cache of sequence %d full (%d of %d)",
                       b, m->P[b], m->Lmax);
  TRY(set_device(m));
  // a draft left by a fused or quadratic cycle belongs to the state those
  // modes carry from cycle to cycle; a cycle of any other mode moves the
  // session on without it
  m->have_draft = false;
  // the cycle runs on the model's stream, after the caller's earlier work
  NDIFF_CUDA_TRY(cudaStreamSynchronize(stream));
  if (!thr) {
    cudaGraphExec_t ge = nullptr;
    TRY(cycle_graph(m, mode, opts->steps, &ge));
    NDIFF_CUDA_TRY(cudaGraphLaunch(ge, m->ms));
    const int rounds = mode == NDIFF_MODE_AR ? 0 : opts->steps;
    return collect(m, mode, rounds + 1, rounds, 0, out_tokens_host, n_out, stats);
  }
  // Threshold sampler: rounds until every sequence's mask word is empty.
  uint32_t tb, rb;
  memcpy(&tb, &opts->tau, 4);
  memcpy(&rb, &opts->tau_revise, 4);
  const float tau = opts->tau, taur = opts->tau_revise;
  const int B = m->B;
  cudaGraphExec_t g_init = nullptr, g_round = nullptr, g_tail = nullptr;
  TRY(cached_graph(m, std::make_tuple((int)PART_INIT, 0, 0, 0u, 0u),
                   [&](cudaStream_t s) {
                     return launch_block_init(m->block_in, m->draft, m->mask, kBlock, m->last_dev,
                                              m->mask_id, B, s);
                   },
                   &g_init));
  TRY(cached_graph(m, std::make_tuple((int)PART_ROUND, 0, 0, tb, rb),
                   [&](cudaStream_t s) {
                     TRY(forward(m, m->block_in, kBlock, 0, FWD_TOKENS, s));
                     return launch_unmask_threshold(m->conf, m->pred, B, kBlock, tau, taur, m->mask,
                                                    m->block_in, m->draft, m->nfixed, m->nrevised,
                                                    s);
                   },
                   &g_round));
  TRY(cached_graph(m, std::make_tuple((int)PART_TAIL, (int)mode, 0, 0u, 0u),
                   [&](cudaStream_t s) { return enqueue_tail(m, mode, s); }, &g_tail));
  NDIFF_CUDA_TRY(cudaGraphLaunch(g_init, m->ms));
  int rounds = 0;
  int64_t revisions = 0;
  int32_t* hmask = m->pin;
  int32_t* hcnt = m->pin + B;  // fixed [B], revised [B]
  for (;;) {
    NDIFF_CUDA_TRY(cudaGraphLaunch(g_round, m->ms));
    NDIFF_CUDA_TRY(cudaMemcpyAsync(hmask, m->mask, (size_t)B * 4, cudaMemcpyDeviceToHost, m->ms));
    NDIFF_CUDA_TRY(cudaMemcpyAsync(hcnt, m->nfixed, (size_t)2 * B * 4, cudaMemcpyDeviceToHost, m->ms));
    TRY(finish(m->ms));
    ++rounds;
    bool open = false;
    for (int b = 0; b < B; ++b) {
      revisions += hcnt[B + b];
      open = open || hmask[b] != 0;
    }
    if (!open) break;
    // every round fixes at least one of each unfinished block's 32 slots
    if (rounds >= kBlock)
      return set_error(NDIFF_ERR_CUDA, "ndiff_decode_step: 32 threshold rounds left slots masked");
  }
  NDIFF_CUDA_TRY(cudaGraphLaunch(g_tail, m->ms));
  return collect(m, mode, rounds + 1, rounds, revisions, out_tokens_host, n_out, stats);
}

ndiff_status ndiff_decode_step_ex(ndiff_model* m, const ndiff_decode_opts* opts,
                                  int32_t* out_tokens_host, int* n_out, ndiff_stats* stats,
                                  cudaStream_t stream) {
  if (!m || !opts || !out_tokens_host || !n_out)
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_decode_step: null pointer");
  *n_out = 0;
  if (m->B != 1)
    return set_error(NDIFF_ERR_UNSUPPORTED,
                     "ndiff_decode_step: batched model; use ndiff_decode_step_batch");
  int32_t n = 0;
  TRY(decode_cycle(m, opts, out_tokens_host, &n, stats, stream));
  *n_out = n;
  return NDIFF_OK;
}

ndiff_status ndiff_decode_step_batch(ndiff_model* m, const ndiff_decode_opts* opts,
                                     int32_t* out_tokens_host, int32_t* n_out_host,
                                     ndiff_stats* stats, cudaStream_t stream) {
  if (!m || !opts || !out_tokens_host || !n_out_host)
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_decode_step_batch: null pointer");
  for (int b = 0; b < m->B; ++b) n_out_host[b] = 0;
  return decode_cycle(m, opts, out_tokens_host, n_out_host, stats, stream);
}

ndiff_status ndiff_decode_step(ndiff_model* m, ndiff_mode mode, int steps, int32_t* out_tokens_host,
                               int* n_out, ndiff_stats* stats, cudaStream_t stream) {
  ndiff_decode_opts o;
  o.mode = mode;
  o.sampler = NDIFF_SAMPLER_TOPK;
  o.steps = steps;
  o.tau = 0.f;
  o.tau_revise = 2.f;
  o.n_cand = 2;  // the quadratic mode's default candidates
  o.cand[0] = 0;
  o.cand[1] = 1;
  return ndiff_decode_step_ex(m, &o, out_tokens_host, n_out, stats, stream);
}

ndiff_status ndiff_model_forward(ndiff_model* m, const int32_t* ids_host, int T, ndiff_mask mode,
                                 float* logits_host, cudaStream_t stream) {
  if (!m || !ids_host) return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_model_forward: null pointer");
  if (m->B != 1)
    return set_error(NDIFF_ERR_UNSUPPORTED, "ndiff_model_forward: batch-1 models only");
  if (T < 1 || T > kBlock)
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_model_forward: 1 <= T <= 32 (got %d)", T);
  if (mode != NDIFF_BIDIR && mode != NDIFF_CAUSAL)
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_model_forward: bad mask mode %d", (int)mode);
  if (m->P[0] + T > m->Lmax)
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_model_forward: KV cache full");
  for (int i = 0; i < T; ++i)
    if (ids_host[i] < 0 || ids_host[i] >= m->V)
      return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_model_forward: token out of range");
  TRY(set_device(m));
  NDIFF_CUDA_TRY(cudaMemcpyAsync(m->ids, ids_host, (size_t)T * 4, cudaMemcpyHostToDevice, stream));
  TRY(forward(m, m->ids, T, mode == NDIFF_CAUSAL ? 1 : 0, FWD_LOGITS, stream));
  if (logits_host)
    NDIFF_CUDA_TRY(cudaMemcpy2DAsync(logits_host, (size_t)m->V * 4, m->logits, (size_t)m->ldl * 4,
                                     (size_t)m->V * 4, T, cudaMemcpyDeviceToHost, stream));
  return finish(stream);
}

ndiff_status ndiff_model_state(const ndiff_model* m, int* kv_len, int32_t* last_token) {
  if (!m) return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_model_state: null model");
  if (kv_len) *kv_len = m->P[0];
  if (last_token) *last_token = m->last[0];
  return NDIFF_OK;
}

ndiff_status ndiff_model_state_batch(const ndiff_model* m, int32_t* kv_len_host,
                                     int32_t* last_host) {
  if (!m) return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_model_state_batch: null model");
  for (int b = 0; b < m->B; ++b) {
    if (kv_len_host) kv_len_host[b] = m->P[b];
    if (last_host) last_host[b] = m->last[b];
  }
  return NDIFF_OK;
}

ndiff_status ndiff_model_read_weight(const ndiff_model* m, int tensor_id, int64_t offset,
                                     int64_t count, float* host_out) {
  if (!m || (!host_out && count > 0))
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_model_read_weight: null pointer");
  const void* base = nullptr;
  int64_t rows = 0, cols = 0, row_off = 0;
  int map = 0;
  bool tiled = false;
  if (!locate(m, tensor_id, &base, &rows, &cols, &row_off, &map, &tiled))
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_model_read_weight: no tensor %d", tensor_id);
  if (offset < 0 || count < 0 || offset + count > rows * cols)
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_model_read_weight: range outside the tensor");
  if (count == 0) return NDIFF_OK;
  TRY(set_device(m));
  float* tmp = nullptr;
  NDIFF_CUDA_TRY(cudaMalloc(&tmp, (size_t)count * 4));
  ndiff_status s = launch_gather_weight(base, m->bf16, cols, row_off, map, tiled, offset, count, tmp, 0);
  if (s == NDIFF_OK) {
    cudaError_t e = cudaMemcpy(host_out, tmp, (size_t)count * 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) s = cuda_error(e, "ndiff_model_read_weight: copy");
  }
  cudaFree(tmp);
  return s;
}

}  // extern "C"
