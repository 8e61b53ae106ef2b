// select.cu — the integer steps of a decode cycle: one warp per sequence for
// the few sequences of a decode step, row-parallel layouts for large batches.
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
//
// Batches of 32-slot blocks take two more layouts, chosen when the row pointers
// are 16-byte aligned:
// unmask_rows_kernel: one thread per sequence, for B >= 256. The CTA stages
//   its 128 rows of conf and pred through shared memory with 16-byte coalesced
//   loads; each thread turns its 32 confidences into order-preserving integer
//   keys (0 marks an unmasked slot) and ranks them with the 496 pairwise
//   comparisons, so no lane exchange is needed; the chosen lists leave through
//   shared memory as one coalesced write. Same selection as unmask_kernel.
// verify32_kernel: one warp per 32 sequences, every global access 16 bytes
//   wide; a warp load covers 4 rows (8 lanes a row), the mismatch bits of a row
//   are OR-ed over its 8 lanes, and the per-sequence results are written by the
//   lane of that sequence.
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

constexpr int ROWS_PER_CTA = 128;
constexpr int UNMASK_ROWS_MIN_B = 256;

// Order-preserving key of a non-NaN float: larger float, larger key; -0 and +0
// share a key so that they tie as float comparison has them tie. Every key is
// >= key(-inf) = 0x007fffff, which leaves 0 free to mark an unmasked slot.
__device__ __forceinline__ uint32_t order_key(float c) {
  uint32_t u = __float_as_uint(c);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(ROWS_PER_CTA)
    unmask_rows_kernel(const float* __restrict__ conf, const int32_t* __restrict__ pred, int B,
                       int k, uint32_t* mask_bits, int32_t* block_in, int32_t* draft,
                       int32_t* chosen) {
  // 16-byte chunk j of row r sits at r * 8 + (j ^ (r & 7)), so the 8 threads of
  // a quarter warp reading chunk j of their own rows hit 8 different bank groups.
  __shared__ int4 s_conf[ROWS_PER_CTA * 8];
  __shared__ int4 s_pred[ROWS_PER_CTA * 8];
  griddep_launch();
  griddep_wait();
  const int row0 = blockIdx.x * ROWS_PER_CTA;
  const int nrows = min(ROWS_PER_CTA, B - row0);
  const int tid = threadIdx.x;
  {
    const int4* gc = reinterpret_cast<const int4*>(conf) + (size_t)row0 * 8;
    const int4* gp = reinterpret_cast<const int4*>(pred) + (size_t)row0 * 8;
    int4 vc[8], vp[8];
#pragma unroll
    for (int it = 0; it < 8; ++it) {
      const int q = it * ROWS_PER_CTA + tid;
      if ((q >> 3) < nrows) {
        vc[it] = __ldg(gc + q);
        vp[it] = __ldg(gp + q);
      }
    }
#pragma unroll
    for (int it = 0; it < 8; ++it) {
      const int q = it * ROWS_PER_CTA + tid;
      const int r = q >> 3, j = q & 7;
      if (r < nrows) {
        s_conf[r * 8 + (j ^ (r & 7))] = vc[it];
        s_pred[r * 8 + (j ^ (r & 7))] = vp[it];
      }
    }
  }
  __syncthreads();
  const bool live = tid < nrows;
  const int b = row0 + tid;
  const uint32_t mask = live ? mask_bits[b] : 0u;
  uint32_t key[32];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int4 v = s_conf[tid * 8 + (j ^ (tid & 7))];
    key[4 * j + 0] = order_key(__int_as_float(v.x));
    key[4 * j + 1] = order_key(__int_as_float(v.y));
    key[4 * j + 2] = order_key(__int_as_float(v.z));
    key[4 * j + 3] = order_key(__int_as_float(v.w));
  }
#pragma unroll
  for (int i = 0; i < 32; ++i) key[i] = ((mask >> i) & 1u) ? key[i] : 0u;
  // rank[i] = number of slots that beat slot i; for i < j, j beats i only on a
  // strictly larger key (ties go to the lower slot). Unmasked slots (key 0)
  // never beat a masked one, and their own ranks are not used.
  int rank[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) rank[i] = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
#pragma unroll
    for (int j = i + 1; j < 32; ++j) {
      const int p = key[j] > key[i] ? 1 : 0;
      rank[i] += p;
      rank[j] += 1 - p;
    }
  }
  __syncthreads();  // every thread holds its keys: s_conf now holds the chosen lists
  int32_t* s_chosen = reinterpret_cast<int32_t*>(s_conf);
  if (live) {
    const int kk = min(k, __popc(mask));
    uint32_t taken = 0u;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int4 v = s_pred[tid * 8 + (j ^ (tid & 7))];
      const int32_t pv4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = 4 * j + e;
        if (key[i] != 0u && rank[i] < kk) {
          draft[(size_t)b * 32 + i] = pv4[e];
          if (i <= 30) block_in[(size_t)b * 32 + i + 1] = pv4[e];
          s_chosen[tid * k + rank[i]] = i;
          taken |= 1u << i;
        }
      }
    }
    for (int r = kk; r < k; ++r) s_chosen[tid * k + r] = -1;
    mask_bits[b] = mask & ~taken;
  }
  __syncthreads();
  int32_t* out = chosen + (size_t)row0 * k;
  for (int q = tid; q < nrows * k; q += ROWS_PER_CTA) out[q] = s_chosen[q];
}

__global__ void __launch_bounds__(128) verify32_kernel(const int32_t* __restrict__ draft,
                                                       const int32_t* __restrict__ target, int B,
                                                       int32_t* accept_len, int32_t* commit,
                                                       int32_t* n_commit, int32_t* kv_len) {
  griddep_launch();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int base = (blockIdx.x * 4 + (threadIdx.x >> 5)) * 32;
  if (base >= B) return;  // uniform over the warp
  const int g = lane >> 3, c = lane & 7;
  const int4* gd = reinterpret_cast<const int4*>(draft);
  const int4* gt = reinterpret_cast<const int4*>(target);
  int4* gc = reinterpret_cast<int4*>(commit);
  int4 d[8], t[8];
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int row = base + it * 4 + g;
    if (row < B) {
      d[it] = __ldg(gd + (size_t)row * 8 + c);
      t[it] = __ldg(gt + (size_t)row * 8 + c);
    } else {
      d[it] = make_int4(0, 0, 0, 0);
      t[it] = d[it];
    }
  }
  int my_len = 32;
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const uint32_t nib = (d[it].x != t[it].x ? 1u : 0u) | (d[it].y != t[it].y ? 2u : 0u) |
                         (d[it].z != t[it].z ? 4u : 0u) | (d[it].w != t[it].w ? 8u : 0u);
    uint32_t bits = nib << (4 * c);
    bits |= __shfl_xor_sync(0xffffffffu, bits, 1);
    bits |= __shfl_xor_sync(0xffffffffu, bits, 2);
    bits |= __shfl_xor_sync(0xffffffffu, bits, 4);
    const int L = bits ? (__ffs(bits) - 1) : 32;
    const int n = min(L + 1, 32);
    const int row = base + it * 4 + g;
    if (row < B) {
      const int s0 = 4 * c;
      gc[(size_t)row * 8 + c] =
          make_int4(s0 + 0 < n ? t[it].x : -1, s0 + 1 < n ? t[it].y : -1,
                    s0 + 2 < n ? t[it].z : -1, s0 + 3 < n ? t[it].w : -1);
    }
    // lane o reports sequence base + o, whose row was loaded in pass o / 4 by
    // lanes 8 * (o % 4) ..
    const int Lo = __shfl_sync(0xffffffffu, L, (lane & 3) * 8);
    if ((lane >> 2) == it) my_len = Lo;
  }
  const int row = base + lane;
  if (row < B) {
    const int n = min(my_len + 1, 32);
    accept_len[row] = my_len;
    n_commit[row] = n;
    if (kv_len) kv_len[row] += n;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0u; }

}  // namespace

ndiff_status launch_unmask(const float* conf, const int32_t* pred, int B, int T, int k,
                           uint32_t* mask_bits, int32_t* block_in, int32_t* draft,
                           int32_t* chosen, cudaStream_t stream) {
  if (B == 0) return NDIFF_OK;
  if (T == 32 && B >= UNMASK_ROWS_MIN_B && aligned16(conf) && aligned16(pred)) {
    NDIFF_CUDA_TRY(launch_k(unmask_rows_kernel, dim3((B + ROWS_PER_CTA - 1) / ROWS_PER_CTA),
                            dim3(ROWS_PER_CTA), 0, stream, conf, pred, B, k, mask_bits, block_in,
                            draft, chosen));
    return NDIFF_OK;
  }
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
  if (T == 32 && aligned16(draft) && aligned16(target) && aligned16(commit)) {
    NDIFF_CUDA_TRY(launch_k(verify32_kernel, dim3((B + 127) / 128), dim3(128), 0, stream, draft,
                            target, B, accept_len, commit, n_commit, kv_len));
    return NDIFF_OK;
  }
  NDIFF_CUDA_TRY(launch_k(verify_kernel, dim3((B + 3) / 4), dim3(128), 0, stream, draft, target, B,
                          T, accept_len, commit, n_commit, kv_len));
  return NDIFF_OK;
}

}  // namespace ndiff
