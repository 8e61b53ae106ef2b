// kernels.h — host-side launchers of libndiff's kernels (internal). Argument
// validation happens in api.cu before any of these is called.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/ndiff.h"

namespace ndiff {

// attn_bf16.cu
int attn_bf16_auto_split(int B, int Hkv, int Lmax);
size_t attn_bf16_workspace(int B, int T, int Hq, int Hkv, int Lmax, int split);
ndiff_status launch_attn_bf16(const void* q, const void* k, const void* v, const int32_t* kv_len,
                              int B, int T, int Hq, int Hkv, int Lmax, int causal, float scale,
                              int split, void* out, void* ws, size_t ws_bytes,
                              cudaStream_t stream);

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
ndiff_status launch_verify_accept(const int32_t* draft, const int32_t* target, int B, int T,
                                  int32_t* accept_len, int32_t* commit, int32_t* n_commit,
                                  int32_t* kv_len, cudaStream_t stream);

}  // namespace ndiff
