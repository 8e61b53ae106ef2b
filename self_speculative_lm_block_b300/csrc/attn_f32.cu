// attn_f32.cu — block-causal attention in fp32 for small head dimensions
// (D <= 64), the tiny model's path. Same visibility rule as the bf16 kernel
// ("Nemotron-Labs-Diffusion: A Tri-Mode Language Model ..." (hotpaper.ai),
// modules: block-wise attention): the whole prefix, plus every block key
// (BIDIR) or the block keys up to the row's slot (CAUSAL).
//
// One warp per (b, slot, head) row. Key j belongs to lane j % 32 at every
// block length, each lane walks its keys in increasing order and the lanes
// merge by a fixed shuffle tree, so a row's result does not depend on T.
#include "common.cuh"
#include "kernels.h"

namespace ndiff {
namespace {

constexpr int MAXD = 64;

__global__ void __launch_bounds__(128) attn_f32_kernel(const float* __restrict__ q,
                                                       const float* __restrict__ kc,
                                                       const float* __restrict__ vc,
                                                       const int32_t* __restrict__ kv_len, int B,
                                                       int T, int Hq, int Hkv, int D, int Lmax,
                                                       int causal, float scale,
                                                       float* __restrict__ out,
                                                       unsigned int* __restrict__ status) {
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= B * T * Hq) return;
  const int h = row % Hq;
  const int t = (row / Hq) % T;
  const int b = row / (Hq * T);
  const int g = h / (Hq / Hkv);
  const int P = checked_prefix(kv_len[b], Lmax - T, status);
  const int nvis = P + (causal ? t + 1 : T);
  const float* qr = q + (size_t)row * D;
  const float* kb = kc + ((size_t)b * Hkv + g) * Lmax * D;
  const float* vb = vc + ((size_t)b * Hkv + g) * Lmax * D;

  // pass 1: the row maximum of the scores
  float m = -INFINITY;
  for (int j = lane; j < nvis; j += 32) {
    float sc = 0.f;
    for (int d = 0; d < D; ++d) sc = fmaf(qr[d], kb[(size_t)j * D + d], sc);
    m = fmaxf(m, sc * scale);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));

  // pass 2: weights, their sum and the weighted values
  float acc[MAXD];
#pragma unroll
  for (int d = 0; d < MAXD; ++d) acc[d] = 0.f;
  float l = 0.f;
  for (int j = lane; j < nvis; j += 32) {
    float sc = 0.f;
    for (int d = 0; d < D; ++d) sc = fmaf(qr[d], kb[(size_t)j * D + d], sc);
    const float pj = expf(sc * scale - m);
    l += pj;
#pragma unroll
    for (int d = 0; d < MAXD; ++d)
      if (d < D) acc[d] = fmaf(pj, vb[(size_t)j * D + d], acc[d]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
#pragma unroll
  for (int d = 0; d < MAXD; ++d) {
    float x = acc[d];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    acc[d] = x;
  }
  const float inv = 1.f / l;
  float* o = out + (size_t)row * D;
#pragma unroll
  for (int d = 0; d < MAXD; ++d)
    if (d < D && (d & 31) == lane) o[d] = acc[d] * inv;
}

}  // namespace

ndiff_status launch_attn_f32(const float* q, const float* k, const float* v,
                             const int32_t* kv_len, int B, int T, int Hq, int Hkv, int D,
                             int Lmax, int causal, float scale, float* out, cudaStream_t stream) {
  const long long rows = (long long)B * T * Hq;
  if (rows == 0) return NDIFF_OK;
  attn_f32_kernel<<<(unsigned)((rows + 3) / 4), 128, 0, stream>>>(q, k, v, kv_len, B, T, Hq, Hkv,
                                                                   D, Lmax, causal, scale, out,
                                                                   device_status_word());
  NDIFF_CUDA_TRY(cudaGetLastError());
  return NDIFF_OK;
}

}  // namespace ndiff
