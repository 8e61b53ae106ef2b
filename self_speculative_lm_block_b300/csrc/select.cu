// select.cu — the two integer steps of a decode cycle, one warp per sequence.
//
// unmask: one denoising round of the 32-token block ("NVIDIA 发布 Nemotron-Labs
//   Diffusion 语言模型系列" (fintech-frontier-insights), "三种生成模式": a block
//   is refined over several rounds). Lane i ranks its slot among the masked
//   slots by (confidence desc, slot asc) with 32 shuffles; the k best are fixed.
// unmask_threshold: the sampler variant whose step count follows the model's
//   confidence ("NVIDIA 发布 Nemotron-Labs Diffusion：三模态语言模型统一 AR 与
//   扩散解码" (aimodeling.com digest of the Hugging Face blog): the refinement
//   steps are a budget, and earlier tokens can be revised). Reading: a round
//   fixes every masked slot with confidence >= tau, or else the single most
//   confident one (ties to the lower slot); before that, a slot fixed in an
//   earlier round takes the new prediction when it differs and its confidence
//   is >= tau_revise. Ballots and one warp argmax per sequence.
// verify_accept: gsyq.cn explainer, §2.3 "自推测解码": accept the agreeing
//   prefix, replace the first mismatch by the verifier's token. One ballot and
//   one find-first-set per sequence.
#include "common.cuh"
#include "kernels.h"

namespace ndiff {
namespace {

__global__ void __launch_bounds__(128) unmask_kernel(const float* __restrict__ conf,
                                                     const int32_t* __restrict__ pred, int B,
                                                     int T, int k, uint32_t* mask_bits,
                                                     int32_t* block_in, int32_t* draft,
                                                     int32_t* chosen) {
  griddep_launch();
  griddep_wait();
  const int b = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int i = threadIdx.x & 31;
  if (b >= B) return;
  const uint32_t valid = (T == 32) ? 0xffffffffu : ((1u << T) - 1u);
  const uint32_t mask = mask_bits[b] & valid;
  const bool masked = (mask >> i) & 1u;
  const float c = (i < T) ? conf[(size_t)b * T + i] : 0.f;
  int rank = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float cj = __shfl_sync(0xffffffffu, c, j);
    const bool mj = (mask >> j) & 1u;
    rank += (mj && (cj > c || (cj == c && j < i))) ? 1 : 0;
  }
  const int cnt = __popc(mask);
  const int kk = min(k, cnt);
  const bool sel = masked && rank < kk;
  if (sel) {
    const int32_t pv = pred[(size_t)b * T + i];
    draft[(size_t)b * T + i] = pv;
    if (i <= T - 2) block_in[(size_t)b * T + i + 1] = pv;
    chosen[(size_t)b * k + rank] = i;
  }
  for (int r = kk + i; r < k; r += 32) chosen[(size_t)b * k + r] = -1;
  const uint32_t taken = __ballot_sync(0xffffffffu, sel);
  if (i == 0) mask_bits[b] = mask & ~taken;
}

__global__ void __launch_bounds__(128)
    unmask_threshold_kernel(const float* __restrict__ conf, const int32_t* __restrict__ pred, int B,
                            int T, float tau, float tau_revise, uint32_t* mask_bits,
                            int32_t* block_in, int32_t* draft, int32_t* n_fixed,
                            int32_t* n_revised) {
  griddep_launch();
  griddep_wait();
  const int b = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int i = threadIdx.x & 31;
  if (b >= B) return;
  const uint32_t valid = (T == 32) ? 0xffffffffu : ((1u << T) - 1u);
  const uint32_t mask = mask_bits[b] & valid;
  const bool in = i < T;
  const bool masked = (mask >> i) & 1u;
  const float c = in ? conf[(size_t)b * T + i] : 0.f;
  const int32_t pv = in ? pred[(size_t)b * T + i] : 0;
  const int32_t dv = in ? draft[(size_t)b * T + i] : 0;
  const bool revise = in && !masked && pv != dv && c >= tau_revise;
  bool fix = masked && c >= tau;
  if (__ballot_sync(0xffffffffu, fix) == 0u && mask != 0u) {
    // no slot reaches tau: the most confident masked slot, lowest on ties
    float bc = masked ? c : -INFINITY;
    int bi = masked ? i : 32;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float oc = __shfl_xor_sync(0xffffffffu, bc, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (oc > bc || (oc == bc && oi < bi)) {
        bc = oc;
        bi = oi;
      }
    }
    fix = (i == bi);
  }
  if (fix || revise) {
    draft[(size_t)b * T + i] = pv;
    if (i <= T - 2) block_in[(size_t)b * T + i + 1] = pv;
  }
  const uint32_t fixed = __ballot_sync(0xffffffffu, fix);
  const uint32_t revised = __ballot_sync(0xffffffffu, revise);
  if (i == 0) {
    mask_bits[b] = mask & ~fixed;
    if (n_fixed) n_fixed[b] = __popc(fixed);
    if (n_revised) n_revised[b] = __popc(revised);
  }
}

__global__ void __launch_bounds__(128) verify_kernel(const int32_t* __restrict__ draft,
                                                     const int32_t* __restrict__ target, int B,
                                                     int T, int32_t* accept_len, int32_t* commit,
                                                     int32_t* n_commit, int32_t* kv_len) {
  griddep_launch();
  griddep_wait();
  const int b = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int i = threadIdx.x & 31;
  if (b >= B) return;
  int32_t tv = 0;
  bool mis = false;
  if (i < T) {
    tv = target[(size_t)b * T + i];
    mis = draft[(size_t)b * T + i] != tv;
  }
  const uint32_t bits = __ballot_sync(0xffffffffu, mis);
  const int L = bits ? (__ffs(bits) - 1) : T;
  const int n = min(L + 1, T);
  if (i < T) commit[(size_t)b * T + i] = (i < n) ? tv : -1;
  if (i == 0) {
    accept_len[b] = L;
    n_commit[b] = n;
    if (kv_len) kv_len[b] += n;
  }
}

}  // namespace

ndiff_status launch_unmask(const float* conf, const int32_t* pred, int B, int T, int k,
                           uint32_t* mask_bits, int32_t* block_in, int32_t* draft,
                           int32_t* chosen, cudaStream_t stream) {
  if (B == 0) return NDIFF_OK;
  NDIFF_CUDA_TRY(launch_k(unmask_kernel, dim3((B + 3) / 4), dim3(128), 0, stream, conf, pred, B, T,
                          k, mask_bits, block_in, draft, chosen));
  return NDIFF_OK;
}

ndiff_status launch_unmask_threshold(const float* conf, const int32_t* pred, int B, int T, float tau,
                                     float tau_revise, uint32_t* mask_bits, int32_t* block_in,
                                     int32_t* draft, int32_t* n_fixed, int32_t* n_revised,
                                     cudaStream_t stream) {
  if (B == 0) return NDIFF_OK;
  NDIFF_CUDA_TRY(launch_k(unmask_threshold_kernel, dim3((B + 3) / 4), dim3(128), 0, stream, conf,
                          pred, B, T, tau, tau_revise, mask_bits, block_in, draft, n_fixed,
                          n_revised));
  return NDIFF_OK;
}

ndiff_status launch_verify_accept(const int32_t* draft, const int32_t* target, int B, int T,
                                  int32_t* accept_len, int32_t* commit, int32_t* n_commit,
                                  int32_t* kv_len, cudaStream_t stream) {
  if (B == 0) return NDIFF_OK;
  NDIFF_CUDA_TRY(launch_k(verify_kernel, dim3((B + 3) / 4), dim3(128), 0, stream, draft, target, B,
                          T, accept_len, commit, n_commit, kv_len));
  return NDIFF_OK;
}

}  // namespace ndiff
