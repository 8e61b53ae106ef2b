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
// unmask_quad_kernel: four lanes per sequence, for B >= 256. Each lane loads
//   8 of the row's confidences with two coalesced 16-byte loads, turns them
//   into order-preserving integer keys (0 marks an unmasked slot). For k <= 8
//   it sorts its eight slots and the k winners are taken one per round, the
//   largest of the four lanes' heads; for larger k it counts for each of its
//   slots the slots that beat it: 28 comparisons among its own and 3 x 64
//   against the keys its three partners pass by shuffle.
//   The lane merges the chosen tokens into its 16-byte chunks of the draft and
//   next-input rows (one shuffle brings the lower lane's last slot for the
//   shift by one) and writes back whole chunks, so no store is a partial
//   sector. Same selection as unmask_kernel, with 4 times the sequences in
//   flight of one thread per sequence and a quarter of the warp-wide shuffles
//   of one warp per sequence.
// verify32_kernel: one warp per 8 sequences (two passes of 4), every global
//   access 16 bytes wide; a warp load covers 4 rows (8 lanes a row), the
//   mismatch bits of a row are OR-ed over its 8 lanes, and the per-sequence
//   results are written by the lane of that sequence. Few rows a warp keeps
//   registers low, so a 65536-sequence batch is resident in one wave.
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

constexpr int QUAD_ROWS_PER_CTA = 32;  // 128 threads, 4 a sequence
constexpr int UNMASK_QUAD_MIN_B = 256;

// Order-preserving key of a non-NaN float: larger float, larger key; -0 and +0
// share a key so that they tie as float comparison has them tie. Every key is
// >= key(-inf) = 0x007fffff, which leaves 0 free to mark an unmasked slot.
__device__ __forceinline__ uint32_t order_key(float c) {
  uint32_t u = __float_as_uint(c);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Four lanes share a sequence; lane q (0..3) owns slots 4q..4q+3 and
// 16+4q..16+4q+3, so each of its two 16-byte loads of a row is coalesced with
// the other lanes' (a warp load covers the first or second half of 8 rows).
__device__ __forceinline__ constexpr int quad_slot(int q, int e) {
  return e < 4 ? 4 * q + e : 16 + 4 * q + (e - 4);
}

// 64-bit xor shuffle.
__device__ __forceinline__ unsigned long long shfl_xor_u64(unsigned long long v, int m) {
  const uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)v, m);
  const uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(v >> 32), m);
  return ((unsigned long long)hi << 32) | lo;
}

// EXTRACT (k <= 8): the k winners are taken one at a time instead of ranking
// every slot. Each lane sorts its eight slots by the composite key
// (key << 5) | (31 - slot), unique per slot and ordered as the selection
// orders slots (larger key first, the lower slot on equal keys), with a
// 19-comparator sorting network; round r then takes the largest head of the
// four lanes' sorted lists (two shuffle-max steps), which is the slot of rank
// r. About half the instructions of the pairwise ranking at k = 8.
template <bool EXTRACT>
__global__ void __launch_bounds__(128, 10)
    unmask_quad_kernel(const float* __restrict__ conf, const int32_t* __restrict__ pred, int B,
                       int k, uint32_t* mask_bits, int32_t* block_in, int32_t* draft,
                       int32_t* chosen) {
  griddep_launch();
  griddep_wait();
  const int q = threadIdx.x & 3;
  const int b = blockIdx.x * QUAD_ROWS_PER_CTA + (threadIdx.x >> 2);
  const bool live = b < B;
  // every lane takes part in the shuffles: a lane past the batch reads row 0
  // (B >= 1) and writes nothing
  const int row = live ? b : 0;
  const int4* gc = reinterpret_cast<const int4*>(conf) + (size_t)row * 8;
  const int4* gp = reinterpret_cast<const int4*>(pred) + (size_t)row * 8;
  const int4 c0 = __ldg(gc + q), c1 = __ldg(gc + 4 + q);
  const int4 p0 = __ldg(gp + q), p1 = __ldg(gp + 4 + q);
  const uint32_t mask = mask_bits[row];
  uint32_t key[8] = {order_key(__int_as_float(c0.x)), order_key(__int_as_float(c0.y)),
                     order_key(__int_as_float(c0.z)), order_key(__int_as_float(c0.w)),
                     order_key(__int_as_float(c1.x)), order_key(__int_as_float(c1.y)),
                     order_key(__int_as_float(c1.z)), order_key(__int_as_float(c1.w))};
  const int32_t pv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
  for (int e = 0; e < 8; ++e) key[e] = ((mask >> quad_slot(q, e)) & 1u) ? key[e] : 0u;
  const int kk = min(k, __popc(mask));
  bool sel[8];
  uint32_t taken = 0u;
  if constexpr (EXTRACT) {
    unsigned long long sk[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) sk[e] = ((unsigned long long)key[e] << 5) | (uint32_t)(31 - quad_slot(q, e));
    constexpr int NET[19][2] = {{0, 1}, {2, 3}, {4, 5}, {6, 7}, {0, 2}, {1, 3}, {4, 6}, {5, 7}, {1, 2}, {5, 6},
                                {0, 4}, {1, 5}, {2, 6}, {3, 7}, {2, 4}, {3, 5}, {1, 2}, {3, 4}, {5, 6}};
#pragma unroll
    for (int c = 0; c < 19; ++c) {  // descending
      const unsigned long long a = sk[NET[c][0]], z = sk[NET[c][1]];
      const bool sw = z > a;
      sk[NET[c][0]] = sw ? z : a;
      sk[NET[c][1]] = sw ? a : z;
    }
    for (int r = 0; r < k; ++r) {  // k <= 8, the same for every lane
      const unsigned long long head = sk[0];
      unsigned long long m = head, o = shfl_xor_u64(m, 1);
      m = o > m ? o : m;
      o = shfl_xor_u64(m, 2);
      m = o > m ? o : m;
      if (r < kk && head == m) {  // this lane holds the slot of rank r
        const int slot = 31 - (int)(m & 31u);
        taken |= 1u << slot;
        if (live) chosen[(size_t)b * k + r] = slot;
#pragma unroll
        for (int e = 0; e < 7; ++e) sk[e] = sk[e + 1];
        sk[7] = 0ull;
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) sel[e] = (taken >> quad_slot(q, e)) & 1u;
  } else {
    // rank[e] = number of slots that beat own slot e: o beats m when
    // key_o + [slot_o < slot_m] > key_m (ties go to the lower slot; the +1 never
    // overflows since every key is <= key(+inf) = 0xff800000).
    int rank[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) rank[e] = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
#pragma unroll
      for (int f = e + 1; f < 8; ++f) {  // own slots rise with e
        const int p = key[f] > key[e] ? 1 : 0;
        rank[e] += p;
        rank[f] += 1 - p;
      }
    }
#pragma unroll
    for (int d = 1; d < 4; ++d) {
      uint32_t o[8];
#pragma unroll
      for (int f = 0; f < 8; ++f) o[f] = __shfl_xor_sync(0xffffffffu, key[f], d);
      // the partner's first-half slots lie below every own second-half slot and
      // its second-half slots above every own first-half slot; within a half
      // the lower lane has the lower slots
      const uint32_t lower = ((q ^ d) < q) ? 1u : 0u;
#pragma unroll
      for (int f = 0; f < 4; ++f) {
        const uint32_t same = o[f] + lower, below = o[f] + 1u;
#pragma unroll
        for (int e = 0; e < 4; ++e) rank[e] += same > key[e] ? 1 : 0;
#pragma unroll
        for (int e = 4; e < 8; ++e) rank[e] += below > key[e] ? 1 : 0;
      }
#pragma unroll
      for (int f = 4; f < 8; ++f) {
        const uint32_t same = o[f] + lower;
#pragma unroll
        for (int e = 0; e < 4; ++e) rank[e] += o[f] > key[e] ? 1 : 0;
#pragma unroll
        for (int e = 4; e < 8; ++e) rank[e] += same > key[e] ? 1 : 0;
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      sel[e] = key[e] != 0u && rank[e] < kk;
      if (sel[e]) taken |= 1u << quad_slot(q, e);
    }
    if (live) {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (sel[e]) chosen[(size_t)b * k + rank[e]] = quad_slot(q, e);
    }
  }
  // block_in[i + 1] takes pred[i]: the first slot of each of the lane's two
  // chunks follows the last slot of the lower lane's chunk (lane 3's first
  // chunk for lane 0's second; nothing for slot 0)
  const int src_lane = (threadIdx.x & ~3) | ((q + 3) & 3);
  const int nb_sel3 = __shfl_sync(0xffffffffu, sel[3] ? 1 : 0, src_lane);
  const int32_t nb_pv3 = __shfl_sync(0xffffffffu, pv[3], src_lane);
  const int nb_sel7 = __shfl_sync(0xffffffffu, sel[7] ? 1 : 0, src_lane);
  const int32_t nb_pv7 = __shfl_sync(0xffffffffu, pv[7], src_lane);
  taken |= __shfl_xor_sync(0xffffffffu, taken, 1);
  taken |= __shfl_xor_sync(0xffffffffu, taken, 2);
  if (!live) return;
  // the draft and next-input chunks are read only now, to keep the selection's
  // registers free (more resident warps hide the extra round of loads)
  int4* gd = reinterpret_cast<int4*>(draft) + (size_t)row * 8;
  int4* gb = reinterpret_cast<int4*>(block_in) + (size_t)row * 8;
  const int4 d0 = gd[q], d1 = gd[4 + q], i0 = gb[q], i1 = gb[4 + q];
  const bool in0 = q > 0 && nb_sel3;
  const bool in4 = q > 0 ? (nb_sel7 != 0) : (nb_sel3 != 0);
  const int32_t v4 = q > 0 ? nb_pv7 : nb_pv3;
  // merged chunks; a chunk is written back only where a slot changed
  const int4 nd0 = make_int4(sel[0] ? pv[0] : d0.x, sel[1] ? pv[1] : d0.y, sel[2] ? pv[2] : d0.z,
                             sel[3] ? pv[3] : d0.w);
  const int4 nd1 = make_int4(sel[4] ? pv[4] : d1.x, sel[5] ? pv[5] : d1.y, sel[6] ? pv[6] : d1.z,
                             sel[7] ? pv[7] : d1.w);
  const int4 ni0 = make_int4(in0 ? nb_pv3 : i0.x, sel[0] ? pv[0] : i0.y, sel[1] ? pv[1] : i0.z,
                             sel[2] ? pv[2] : i0.w);
  const int4 ni1 = make_int4(in4 ? v4 : i1.x, sel[4] ? pv[4] : i1.y, sel[5] ? pv[5] : i1.z,
                             sel[6] ? pv[6] : i1.w);
  if (sel[0] || sel[1] || sel[2] || sel[3]) gd[q] = nd0;
  if (sel[4] || sel[5] || sel[6] || sel[7]) gd[4 + q] = nd1;
  if (in0 || sel[0] || sel[1] || sel[2]) gb[q] = ni0;
  if (in4 || sel[4] || sel[5] || sel[6]) gb[4 + q] = ni1;
  for (int r = kk + q; r < k; r += 4) chosen[(size_t)b * k + r] = -1;
  if (q == 0) mask_bits[b] = mask & ~taken;
}

constexpr int VERIFY_PASSES = 2;                   // rows a warp takes: 4 per pass
constexpr int VERIFY_ROWS_PER_WARP = 4 * VERIFY_PASSES;

__global__ void __launch_bounds__(128) verify32_kernel(const int32_t* __restrict__ draft,
                                                       const int32_t* __restrict__ target, int B,
                                                       int32_t* accept_len, int32_t* commit,
                                                       int32_t* n_commit, int32_t* kv_len) {
  griddep_launch();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int base = (blockIdx.x * 4 + (threadIdx.x >> 5)) * VERIFY_ROWS_PER_WARP;
  if (base >= B) return;  // uniform over the warp
  const int g = lane >> 3, c = lane & 7;
  const int4* gd = reinterpret_cast<const int4*>(draft);
  const int4* gt = reinterpret_cast<const int4*>(target);
  int4* gc = reinterpret_cast<int4*>(commit);
  int4 d[VERIFY_PASSES], t[VERIFY_PASSES];
#pragma unroll
  for (int it = 0; it < VERIFY_PASSES; ++it) {
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
  for (int it = 0; it < VERIFY_PASSES; ++it) {
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
    // lane o < VERIFY_ROWS_PER_WARP reports sequence base + o, whose row was
    // loaded in pass o / 4 by lanes 8 * (o % 4) ..
    const int Lo = __shfl_sync(0xffffffffu, L, (lane & 3) * 8);
    if ((lane >> 2) == it) my_len = Lo;
  }
  const int row = base + lane;
  if (lane < VERIFY_ROWS_PER_WARP && row < B) {
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
  if (T == 32 && B >= UNMASK_QUAD_MIN_B && aligned16(conf) && aligned16(pred) &&
      aligned16(draft) && aligned16(block_in)) {
    NDIFF_CUDA_TRY(launch_k(k <= 8 ? unmask_quad_kernel<true> : unmask_quad_kernel<false>,
                            dim3((B + QUAD_ROWS_PER_CTA - 1) / QUAD_ROWS_PER_CTA), dim3(128), 0,
                            stream, conf, pred, B, k, mask_bits, block_in, draft, chosen));
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
    const int rows_per_cta = 4 * VERIFY_ROWS_PER_WARP;
    NDIFF_CUDA_TRY(launch_k(verify32_kernel, dim3((B + rows_per_cta - 1) / rows_per_cta),
                            dim3(128), 0, stream, draft, target, B, accept_len, commit, n_commit,
                            kv_len));
    return NDIFF_OK;
  }
  NDIFF_CUDA_TRY(launch_k(verify_kernel, dim3((B + 3) / 4), dim3(128), 0, stream, draft, target, B,
                          T, accept_len, commit, n_commit, kv_len));
  return NDIFF_OK;
}

}  // namespace ndiff
