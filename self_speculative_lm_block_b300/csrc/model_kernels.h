// model_kernels.h — host launchers of the model's small kernels (internal).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"

namespace ndiff {

// Storage row of logical row r of a bf16 weight tensor, chosen so that the two
// rows a projection epilogue combines sit next to each other in one 128-row
// tile: gate row j -> (j/64)*128 + 2(j%64), up row j -> the row after it;
// in a q or k head of 128 rows, dim i < 64 -> 2i and dim i + 64 -> 2i + 1
// (the rotate-half RoPE pair). fp32 models store every tensor as is.
enum { ROWMAP_IDENTITY = 0, ROWMAP_GATE = 1, ROWMAP_UP = 2, ROWMAP_ROPE = 3 };

// tiled: the weight is stored as contiguous 128 x 64 tiles (see store_index).
ndiff_status launch_init_normal(void* dst, bool bf16, int tensor_id, int64_t rows, int64_t cols,
                                int64_t row_off, int map, bool tiled, uint64_t seed, double sigma,
                                cudaStream_t s);
ndiff_status launch_gather_weight(const void* src, bool bf16, int64_t cols, int64_t row_off,
                                  int map, bool tiled, int64_t offset, int64_t count, float* out,
                                  cudaStream_t s);
ndiff_status launch_rope_table(float2* tab, int Lmax, int D, double base, cudaStream_t s);
ndiff_status launch_embed(const void* E, bool bf16, const int32_t* ids, int T, int V, int d,
                          float* x, cudaStream_t s);
// The unsummed partial tiles of a GEMM_EPI_PARTIAL projection of mt token
// columns: the workspace and the stream-K partition (U k-steps over G CTAs,
// nks k-steps a tile, maxseg slots a CTA).
struct PartialPlan {
  const float* part;
  int nks, U, G, maxseg;
};

// x += the projection's summed partials, then h = bf16(RMSNorm(x)), for token
// rows 0..T-1 (the output / down projection and the norm after it).
ndiff_status launch_residual_rmsnorm(float* x, int T, int d, float eps, __nv_bfloat16* h,
                                     const PartialPlan& pp, int mt, cudaStream_t s);
// act = SwiGLU of the summed gate/up partials (ntile 128-row tiles).
ndiff_status launch_swiglu_merge(const PartialPlan& pp, int ntile, int T, __nv_bfloat16* act, int64_t lda,
                                 int mt, cudaStream_t s);
// q and the block's K/V cache rows from the summed QKV partials (RoPE on q and
// k; positions / cache rows kv_len[0] + m, or per 32-row block from blk_pos).
ndiff_status launch_qkv_merge(const PartialPlan& pp, int T, int Hq, int Hkv, int Lmax,
                              const int32_t* kv_len, const int32_t* blk_pos, const float2* rope,
                              __nv_bfloat16* q, __nv_bfloat16* kc, __nv_bfloat16* vc, int mt,
                              cudaStream_t s);
ndiff_status launch_rmsnorm(const float* x, int T, int d, float eps, void* out, bool bf16,
                            cudaStream_t s);
ndiff_status launch_linear_f32(const float* x, int ldx, const float* W, int N, int K, float* y,
                               int ldy, int T, cudaStream_t s);
ndiff_status launch_qkv_rope_f32(const float* y, int T, int Hq, int Hkv, int D, int Lmax,
                                 const int32_t* kv_len, const float2* rope, float* qb, float* kc,
                                 float* vc, cudaStream_t s);
ndiff_status launch_swiglu_f32(const float* y, int T, int ffn, float* a, cudaStream_t s);
ndiff_status launch_resid_add_f32(float* x, const float* y, int n, cudaStream_t s);
// B sequences: block_in / draft [B][T], mask [B], last [B].
ndiff_status launch_block_init(int32_t* block_in, int32_t* draft, uint32_t* mask, int T,
                               const int32_t* last, int32_t mask_id, int B, cudaStream_t s);
// B sequences: tokens [B][stride], n_ptr [B] (or n_const), last / kv_len [B].
ndiff_status launch_commit(const int32_t* tokens, int stride, const int32_t* n_ptr, int n_const,
                           int kv_add, int32_t* last, int32_t* kv_len, int B, cudaStream_t s);
ndiff_status launch_set_token(int32_t* ids, int32_t tok, cudaStream_t s);
ndiff_status launch_kv_add(int32_t* kv_len, int add, cudaStream_t s);
// Fused verify + draft forward (one sequence): its 64 input tokens and the
// draft half's prefix; after verification, the next draft when all 32 drafts
// were accepted.
ndiff_status launch_fused_input(int32_t* fin, const int32_t* block_in, const int32_t* draft,
                                int32_t mask_id, const int32_t* kv_len, int32_t* kv_len2,
                                cudaStream_t s);
// Quadratic forward (one sequence, 128 rows): its input, the candidate
// blocks' prefixes / key remaps / positions, and the stash of the draft of the
// verified acceptance length.
ndiff_status launch_quad_input(int32_t* fin, const int32_t* block_in, const int32_t* draft,
                               int32_t mask_id, const int32_t* kv_len, const int32_t* cand,
                               int32_t* kvc, int4* remap, int32_t* blk_pos, cudaStream_t s);
ndiff_status launch_quad_stash(const int32_t* pred, const int32_t* acclen, const int32_t* cand,
                               const int32_t* last, int32_t* draft, int32_t* block_in,
                               cudaStream_t s);
ndiff_status launch_fused_stash(const int32_t* pred2, const int32_t* acclen, const int32_t* last,
                                int32_t* draft, int32_t* block_in, cudaStream_t s);

}  // namespace ndiff
