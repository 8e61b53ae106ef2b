// kernels.h — host-side launchers of libndiff's kernels (internal). Argument
// validation happens in api.cu before any of these is called.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/ndiff.h"

namespace ndiff {

// api.cu: the argument checks of ndiff_block_attn (every entry point of block
// attention runs them before anything else), and the CUDA context current on
// the calling thread (nullptr if none), which keys the caches of device
// addresses: a cudaDeviceReset or another context makes a cached address stale.
ndiff_status check_block_attn_args(ndiff_dtype dt, const void* q, const void* k, const void* v,
                                   const int32_t* kv_len, int B, int T, int Hq, int Hkv, int D,
                                   int Lmax, ndiff_mask mode, const void* out);
void* current_context();

// attn_bf16.cu
int attn_bf16_auto_split(int B, int Hkv, int Lmax);
size_t attn_bf16_workspace(int B, int T, int Hq, int Hkv, int Lmax, int split);
// remap (device, [B] {x, S, cache index, 0}, nullptr = none): sequence b reads
// cache `cache index` (of ncache caches) and finds its virtual keys >= x (a
// multiple of 64, at most kv_len) at cache rows S (a multiple of 64) + key - x;
// the prefix rows [x, kv_len) are copied there by the kernel. Needs
// S + (kv_len - x) + T + 63 < Lmax. x = kNoRemap: no moved keys, only the
// cache index applies. Entries outside this contract are reported as bad
// input and ignored.
constexpr int kNoRemap = 0x7fffffc0;

ndiff_status launch_attn_bf16(const void* q, const void* k, const void* v, const int32_t* kv_len,
                              int B, int T, int Hq, int Hkv, int Lmax, int causal, float scale,
                              int split, void* out, void* ws, size_t ws_bytes,
                              cudaStream_t stream, const int4* remap = nullptr, int ncache = 0,
                              int early_kv = 0, const void* l2pf = nullptr, size_t l2pf_bytes = 0,
                              const void* rpf = nullptr, int rpf_U = 0, int rpf_G = 0);

// attn_f32.cu
ndiff_status launch_attn_f32(const float* q, const float* k, const float* v,
                             const int32_t* kv_len, int B, int T, int Hq, int Hkv, int D,
                             int Lmax, int causal, float scale, float* out, cudaStream_t stream);

// reduce.cu
ndiff_status launch_logits_reduce(ndiff_dtype dt, const void* logits, int R, int V, int64_t ld,
                                  int exclude_id, int32_t* argmax, float* conf,
                                  cudaStream_t stream);

// select.cu
ndiff_status launch_unmask(const float* conf, const int32_t* pred, int B, int T, int k,
                           uint32_t* mask_bits, int32_t* block_in, int32_t* draft,
                           int32_t* chosen, cudaStream_t stream);
ndiff_status launch_unmask_threshold(const float* conf, const int32_t* pred, int B, int T, float tau,
                                     float tau_revise, uint32_t* mask_bits, int32_t* block_in,
                                     int32_t* draft, int32_t* n_fixed, int32_t* n_revised,
                                     cudaStream_t stream);
ndiff_status launch_verify_accept(const int32_t* draft, const int32_t* target, int B, int T,
                                  int32_t* accept_len, int32_t* commit, int32_t* n_commit,
                                  int32_t* kv_len, cudaStream_t stream);

// gemm_bf16.cu — y = x W^T for at most 32 token rows, with fused epilogues
// GEMM_EPI_PARTIAL (weight-streaming kernel): segment s of CTA c (its part of
// one tile; s counts from 0 in k order) stores its partial tile at
// ws[((c * maxseg + s) * MT + m) * 128 + r] (token row m, tile row r) and does
// nothing else; a consumer kernel adds a tile's partials in contributor order
// (partial_slot gives contributor c's segment index for tile t).
enum { GEMM_EPI_F32 = 0, GEMM_EPI_RESID = 1, GEMM_EPI_SWIGLU = 2, GEMM_EPI_QKV = 3, GEMM_EPI_ARGMAX = 4,
       GEMM_EPI_PARTIAL = 5 };

struct GemmParams {
  int N, T, mode;          // weight rows, valid token rows (<= 32), epilogue
  int w_tiled;             // W stored as contiguous 128 x 64 tiles (else row-major)
  int S, nks, items;       // wide kernel: K splits, 64-wide K steps, work items (set by the launcher)
  int ntiles;              // weight-streaming kernel: 128-row tiles (set by the launcher)
  int maxseg;              // GEMM_EPI_PARTIAL: segment slots per CTA (gemm_plan_maxseg)
  float* ws;               // weight-streaming kernel: partial tiles [grid][2][128][MT] fp32
  int* counters;           // [tiles] arrival counters, zero between launches
  unsigned int* status;    // device status word
  float* out;              // F32: out[m*ldo + n] = y; RESID: out[m*ldo + n] += y
  int64_t ldo;
  __nv_bfloat16* act;      // SWIGLU: act[m*lda + j] = silu(gate_j) * up_j
  int64_t lda;
  __nv_bfloat16* q;        // QKV: q [T][Hq][128]; k/v caches [Hkv][Lmax][128]
  __nv_bfloat16* kc;
  __nv_bfloat16* vc;
  int Hq, Hkv, Lmax;
  const int32_t* kv_len;   // QKV: committed prefix (batch 1)
  const float2* rope;      // QKV: (cos, sin) [Lmax][64]
  float4* red;             // ARGMAX: per (tile, token row) (max, sum of exp(y - max),
                           // best allowed value, its id as int bits) [tiles][32]
  int excl;                // ARGMAX: id left out of the argmax (-1: none)
  int Tb;                  // wide kernel, QKV: tokens per sequence (token m is slot m % Tb
                           // of sequence m / Tb; caches [B][Hkv][Lmax][128], kv_len [B])
  const int32_t* blk_pos;  // QKV, weight-streaming kernel (nullptr: token row m has position
                           // and cache row kv_len[0] + m): {position, cache row} of the first
                           // row of each 32-row block [MT/32][2]
};

// Weight-streaming kernel: a stream-K partition of the ntiles * nks k-steps
// over `grid` CTAs (S unused, items = ntiles). Wide kernel: items of (tile,
// token chunk), S = 1.
struct GemmPlan {
  int ntiles, nks, S, items, grid;
  int nchunks;             // wide kernel: 256-row token chunks (1 for the skinny kernel)
};

// The weight-streaming projection for mt = 32 token rows (a block, or one
// token), mt = 64 (two blocks: the fused verify + draft forward) or mt = 128
// (four blocks: the quadratic forward). The stream-K partition depends on
// (N, K, grid) only, so a row's arithmetic is the same for every row count
// and every mt.
GemmPlan gemm_plan(int N, int K);
// Most segments (tiles touched) of one CTA's run of k-steps under the plan.
int gemm_plan_maxseg(const GemmPlan& pl);
// GEMM_EPI_PARTIAL workspace: [grid][maxseg][mt][128] fp32.
size_t gemm_partial_only_bytes(const GemmPlan& pl, int mt);
size_t gemm_partials_bytes(const GemmPlan& pl, int mt = 32);
ndiff_status gemm_make_maps(const void* w, int N, int K, bool w_tiled, const void* x, int M,
                            CUtensorMap* tmW, CUtensorMap* tmX, int mt = 32);
ndiff_status launch_gemm_bf16(const CUtensorMap& tmW, const CUtensorMap& tmX, const GemmPlan& pl,
                              GemmParams p, cudaStream_t stream, int mt = 32);
// Merges the per-tile partials of a GEMM_EPI_ARGMAX launch (red[tile * stride
// + t]): argmax[t] and the softmax probability conf[t] of that id for token
// rows t < T.
ndiff_status launch_argmax_merge(const float4* red, int ntiles, int T, int stride, int32_t* argmax,
                                 float* conf, cudaStream_t stream);

// The projection for any number of token rows M (several sequences): items of
// (128-row weight tile, token chunk), no K split; chunks of 64 rows (tcgen05
// M128 N64) when M <= 64, else of 256 rows (M128 N256). The X map's box must
// have that many rows (gemm_wide_make_xmap with box_rows = 64 or 256); W maps
// as gemm_make_maps.
GemmPlan gemm_wide_plan(int N, int K, int M);
inline int gemm_wide_box_rows(int M) { return M <= 64 ? 64 : 256; }
ndiff_status gemm_wide_make_xmap(const void* x, int M, int K, CUtensorMap* tmX, int box_rows = 256);
ndiff_status launch_gemm_wide(const CUtensorMap& tmW, const CUtensorMap& tmX, const GemmPlan& pl,
                              GemmParams p, cudaStream_t stream);

}  // namespace ndiff
