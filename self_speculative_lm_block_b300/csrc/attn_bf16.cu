// attn_bf16.cu — block-causal GQA attention over a bf16 KV cache on sm_103a.
//
// Operation ("Nemotron-Labs-Diffusion: A Tri-Mode Language Model ..." (hotpaper.ai),
// technical approach / modules: block-wise attention; "NVIDIA 发布 Nemotron-Labs
// Diffusion 语言模型系列" (fintech-frontier-insights), "三种生成模式": 32-token
// blocks; "训练路线": block-wise attention that keeps the KV cache usable):
//   out[b][i][h] = softmax_j(scale * q[b][i][h].k[b][g][j]) . v[b][g][j]
// over the committed prefix j < P_b plus the block keys P_b + t, t < T (BIDIR)
// or t <= i (CAUSAL).
//
// Design (one CTA per (batch b, kv head g, KV split s)):
//   * The G = Hq/Hkv query heads of kv head g and the T block slots form one
//     128-row tile (row r = t*G + hh), so each K/V tile streamed from HBM feeds
//     all G heads: S = Q K^T and O += P V are 128 x 64 x 128 and 128 x 128 x 64
//     tcgen05 MMAs with fp32 accumulators in TMEM (O: 128 columns, S: two
//     64-column buffers).
//   * Warp 0 streams Q once and K/V tiles of 64 keys through a 4-stage TMA
//     ring (128-byte swizzle); warp 1 issues the MMAs; warps 2-5 (one TMEM lane
//     quarter each, one thread per row) run the online softmax in the log2
//     domain, write P as bf16 into shared memory and rescale O in TMEM only
//     when the running maximum grows by more than 2^8 (the final normalisation
//     uses the same stale maximum, so the result is unchanged).
//   * KV splits sit at absolute key positions (multiples of the split length),
//     and masked keys contribute exact zeros, so a row's result does not
//     depend on T: a CAUSAL block of T rows reproduces T single-row calls.
//   * Splits of one (b, g) are merged by attn_combine (log-sum-exp weights).
//   * Remapped keys (the draft blocks of quadratic self-speculation): a
//     sequence may read the cache of another (all candidate blocks share the
//     verified sequence's cache) and may move its virtual keys from a
//     64-aligned position x on to a 64-aligned scratch row S of that cache, so
//     that a block can follow a prefix of any length without overwriting the
//     cache rows past it. The rows [x, P) of the prefix that share x's tile are
//     copied to S by the one CTA that reads that tile, before its loads.
//   * Every mbarrier wait is bounded; on expiry the CTA records a timeout in
//     the device status word, drains its TMA loads, frees TMEM and exits.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace ndiff {
namespace attn {

constexpr int BN = 64;      // keys per tile
constexpr int NST = 6;      // K/V pipeline stages
constexpr int ROWS = 128;   // MMA M (G * T rows)
constexpr int DH = 128;     // head dim
constexpr int KT_BYTES = BN * DH * 2;    // 16 KB: two halves of 8 KB
constexpr int P_BYTES = ROWS * BN * 2;   // 16 KB
constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + NST * KT_BYTES;
constexpr int OFF_P = OFF_V + NST * KT_BYTES;
// (m, l) of both softmax groups at the end, in the P buffers (free by then)
constexpr int OFF_ML = OFF_P;
constexpr int OFF_BAR = OFF_P + 2 * P_BYTES;
constexpr int N_BARS = 1 + 3 * NST + 2 * 3 + 2 + 2 + 1;
constexpr int SMEM_BYTES = OFF_BAR + N_BARS * 8 + 64 + 1024;
// TMEM columns: O of softmax group 0 [0,128), of group 1 [128,256), Q as the
// S product's A operand [256,320) (two bf16 per column), three 64-column S
// buffers [320,512) (tile j uses buffer j % 3).
constexpr int TMEM_COLS = 512;
constexpr int TQ = 256;
constexpr int TS = 320;
constexpr int NSB = 3;
constexpr int THREADS = 320;                       // producer, MMA, 2 x 4 softmax warps
constexpr float RESCALE_THRESHOLD = 8.0f;          // log2 units
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");

struct Params {
  const __nv_bfloat16* q;  // [B][T][Hq][128]
  const int32_t* kv_len;
  int B, T, Hq, Hkv, G, Lmax;
  float scale_log2;   // scale * log2(e)
  int causal;
  int split;          // keys per split (multiple of BN)
  int nsplit_max;     // splits per (b, g) in the grid
  __nv_bfloat16* out;
  const __nv_bfloat16* kc;  // the caches (for the remapped-key copy)
  const __nv_bfloat16* vc;
  float* ws_o;        // [B][Hkv][nsplit_max][128][128]
  float2* ws_ml;      // [B][Hkv][nsplit_max][128]
  const int32_t* order;  // [B * nsplit_max] items (b * nsplit_max + split), longest first;
                         // nullptr: the grid is (nsplit_max, Hkv, B) in natural order
  const int4* remap;     // per sequence {x, S, cache index, 0}: virtual keys >= x sit at
                         // cache rows S + (key - x) of that cache; nullptr: none
  int ncache;            // caches behind k/v when remap is set
  const char* l2pf;      // nullptr, or bytes (the next projection's weights) that the CTAs prefetch
  size_t l2pf_bytes;     // into L2 between them once their own K/V loads are out
  const char* rpf;       // nullptr, or a stream-K projection's weights (tiled, 16 KB a k-step):
  int rpf_U, rpf_G;      // of each of its G runs of U / G k-steps, k-steps [6, 12) past the run's
                         // start (the projection's CTAs load the first six themselves)
  int early_kv;          // 1: kv_len is final when the kernel starts (the previous kernel
                         // triggers its dependents only after its own wait), so the prefix
                         // K/V tiles stream before griddepcontrol.wait; q and the block's own
                         // K/V rows are read after it
  unsigned int* status;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// (lo, hi) -> bf16x2 with lo in the low half, round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b, float& sa, float& sb) {
  __nv_bfloat16 ha = __float2bfloat16_rn(a), hb = __float2bfloat16_rn(b);
  sa = __bfloat162float(ha);
  sb = __bfloat162float(hb);
  return (uint32_t)__bfloat16_as_ushort(ha) | ((uint32_t)__bfloat16_as_ushort(hb) << 16);
}

// Warp-uniform bounded wait: every lane polls, the warp agrees on the result
// (tcgen05.ld/st that follow are warp-collective).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, unsigned int* status,
                                          volatile int* abort_flag) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, status, abort_flag));
}

// Waits that ignore the abort flag (used to drain TMA loads before exit).
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t b = smem_u32(bar);
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(b, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) return;
  }
}

// Named barrier of the 256 softmax threads (both groups).
__device__ __forceinline__ bool softmax_bar_and(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 256, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}

// Named barrier `id` of the 128 threads of one softmax group; returns the AND
// of `pred` over them.
__device__ __forceinline__ bool group_bar_and(int id, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id)
      : "memory");
  return r != 0;
}

__global__ void __launch_bounds__(THREADS, 1)
    attn_bf16_kernel(const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  if (!p.early_kv) griddep_wait();
  int s_idx = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  if (p.order != nullptr) {  // 1-D grid: item rank * Hkv + kv head
    const int item = p.order[blockIdx.x / p.Hkv];
    g = blockIdx.x % p.Hkv;
    b = item / p.nsplit_max;
    s_idx = item % p.nsplit_max;
  }
  const int P = checked_prefix(p.kv_len[b], p.Lmax - p.T, p.status);
  int cb = b, rx = 0x7fffffff, rs = 0;
  if (p.remap != nullptr) {
    const int4 rm = p.remap[b];
    // an entry outside its contract (64-aligned x <= P and S, room for the
    // moved keys, an existing cache) is reported and ignored
    const bool ok = rm.z >= 0 && rm.z < p.ncache && rm.y >= 0 && (rm.y & 63) == 0 &&
                    (rm.x & 63) == 0 && rm.x >= 0 && (rm.x == 0x7fffffc0 ||
                    (rm.x <= P && rm.y + (P - rm.x) + p.T + 63 < p.Lmax));
    if (ok) {
      rx = rm.x;
      rs = rm.y;
      cb = rm.z;
    } else if (threadIdx.x == 0) {
      atomicOr(p.status, kStatusBadInput);
    }
    if (!ok) cb = b < p.ncache ? b : 0;
  }
  const int nkeys = P + p.T;
  const int k_begin = s_idx * p.split;
  if (k_begin >= nkeys) {  // this split is past the sequence (uniform per CTA)
    if (p.early_kv) griddep_wait();
    return;
  }
  const int k_end = min(k_begin + p.split, nkeys);
  const int ntiles = (k_end - k_begin + BN - 1) / BN;
  const int nsplit_b = (nkeys + p.split - 1) / p.split;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* v_full = k_full + NST;
  uint64_t* kv_empty = v_full + NST;
  uint64_t* s_full = kv_empty + NST;   // [NSB] S product of the buffer landed
  uint64_t* s_free = s_full + NSB;     // [NSB] S buffer read by its softmax group
  uint64_t* o_done = s_free + NSB;     // [2] PV products of a group completed
  uint64_t* g_done = o_done + 2;       // [2] drain of a group's PV products at exit
  uint64_t* mma_done = g_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + N_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float2* ml = reinterpret_cast<float2*>(smem + OFF_ML);  // [2][128] (m, l) per group

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    mbar_init(q_full, 128);
    for (int i = 0; i < NST; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < NSB; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 128);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&o_done[i], 1);
      mbar_init(&g_done[i], 1);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_launch();
  const uint32_t tmem = *tmem_slot;

  uint8_t* sK = smem + OFF_K;
  uint8_t* sV = smem + OFF_V;
  uint8_t* sP = smem + OFF_P;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    const int row0 = (cb * p.Hkv + g) * p.Lmax;
    if (rx >= k_begin && rx < k_end && rx < P) {
      // this CTA reads the tile at x: copy its prefix rows [x, P) to S first
      // (generic-proxy stores, then a proxy fence before the TMA loads)
      const int nrow = P - rx;
      for (int e = lane; e < 2 * nrow * 16; e += 32) {
        const int which = e / (nrow * 16), rem = e % (nrow * 16);
        const int row = rem / 16, c16 = rem % 16;
        const __nv_bfloat16* base = which ? p.vc : p.kc;
        const uint4 val = reinterpret_cast<const uint4*>(base + ((size_t)row0 + rx + row) * DH)[c16];
        reinterpret_cast<uint4*>(const_cast<__nv_bfloat16*>(base) + ((size_t)row0 + rs + row) * DH)[c16] =
            val;
      }
      asm volatile("fence.proxy.async.global;" ::: "memory");
      __syncwarp();
    }
    if (lane == 0) {
      int issued = 0;
      // early_kv: the tiles of prefix keys (written by earlier steps) that fit
      // the ring go out before the wait for the previous kernel
      const int npre = !p.early_kv ? 0 : min(min(ntiles, NST), max(0, (P - k_begin) / BN));
      const uint64_t kvpol = l2_evict_first_policy();  // K/V: read once per step
      for (int j = 0; j < ntiles; ++j) {
        if (j == npre && p.early_kv) griddep_wait();
        const int st = j % NST, use = j / NST;
        if (use > 0 && !mbar_wait(&kv_empty[st], (use - 1) & 1, p.status, abort_flag)) break;
        const int vkey = k_begin + j * BN;
        const int key = row0 + (vkey >= rx ? rs + (vkey - rx) : vkey);
        uint8_t* dk = sK + st * KT_BYTES;
        uint8_t* dv = sV + st * KT_BYTES;
        mbar_arrive_expect_tx(&k_full[st], KT_BYTES);
        tma_load_2d_hint(dk, &tmK, &k_full[st], 0, key, kvpol);
        tma_load_2d_hint(dk + 8192, &tmK, &k_full[st], 64, key, kvpol);
        mbar_arrive_expect_tx(&v_full[st], KT_BYTES);
        tma_load_2d_hint(dv, &tmV, &v_full[st], 0, key, kvpol);
        tma_load_2d_hint(dv + 8192, &tmV, &v_full[st], 64, key, kvpol);
        issued = j + 1;
      }
      if (p.l2pf != nullptr) {
        // A decode step's attention leaves HBM mostly idle (a few MB of K/V):
        // the CTAs pull the output projection's weights into L2 meanwhile, in
        // 64 KB bulk prefetches, an equal slice each.
        const int nct = gridDim.x * gridDim.y * gridDim.z;
        const int cid = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
        const size_t per = ((p.l2pf_bytes + nct - 1) / nct + 65535) & ~(size_t)65535;
        const size_t b0 = per * cid, b1 = b0 + per < p.l2pf_bytes ? b0 + per : p.l2pf_bytes;
        for (size_t o = b0; o < b1; o += 65536) {
          const uint32_t n = (uint32_t)(b1 - o < 65536 ? b1 - o : 65536);
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.l2pf + o), "r"(n) : "memory");
        }
        if (p.rpf != nullptr) {
          for (int c = cid; c < p.rpf_G; c += nct) {
            const int s0 = (int)((long long)c * p.rpf_U / p.rpf_G);
            const int s1 = (int)((long long)(c + 1) * p.rpf_U / p.rpf_G);
            const int k0 = s0 + 6, k1 = min(s1, k0 + 6);
            if (k1 > k0)
              asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.rpf + (size_t)k0 * 16384),
                           "r"((uint32_t)(k1 - k0) * 16384u) : "memory");
          }
        }
      }
      if (*abort_flag) {
        // Let every issued copy land before the CTA's shared memory goes away.
        for (int j = (issued > NST ? issued - NST : 0); j < issued; ++j) {
          mbar_drain(&k_full[j % NST], (j / NST) & 1);
          mbar_drain(&v_full[j % NST], (j / NST) & 1);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S issuer
    // S(j) = Q K_j^T into buffer j % NSB once K_j landed and the group that
    // read S(j - NSB) released the buffer. PV products are issued by the
    // softmax groups themselves.
    if (lane == 0) {
      const uint32_t idS = idesc_bf16_f32(ROWS, BN, false, false);
      const uint32_t ka = smem_u32(sK);
      bool ok = mbar_wait(q_full, 0, p.status, abort_flag);
      tc_fence_after();
      for (int j = 0; ok && j < ntiles; ++j) {
        const int st = j % NST, sb = j % NSB;
        if (j >= NSB && !mbar_wait(&s_free[sb], ((j / NSB) - 1) & 1, p.status, abort_flag)) break;
        if (!mbar_wait(&k_full[st], (j / NST) & 1, p.status, abort_flag)) break;
        tc_fence_after();
        const uint32_t kb = ka + st * KT_BYTES;
        const uint32_t dS = tmem + TS + sb * 64;
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const uint32_t off = (kk & 3) * 32;
          const uint64_t bd = smem_desc_sw128(kb + (kk >> 2) * 8192 + off, 16, 1024);
          umma_f16_ts(dS, tmem + TQ + kk * 8, bd, idS, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[sb]);
      }
      umma_commit(mma_done);
      mbar_drain(mma_done, 0);
    }
  } else {
    // ------------------------------------------------- softmax, two groups
    // Group w takes the tiles j with j % 2 == w and keeps its own running
    // maximum, sum and O accumulator; the two are merged at the end. After
    // writing P(j) the group's first thread issues O_w += P(j) V_j itself.
    const int grp = (warp - 2) >> 2;            // 0 or 1
    const uint32_t quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const bool valid = r < p.G * p.T;
    const int t = r / p.G;
    const int vis_end = valid ? P + (p.causal ? t + 1 : p.T) : 0;
    const uint32_t tl = tmem + ((quarter * 32u) << 16);
    const uint32_t tO = tl + grp * DH;
    const int tid128 = (threadIdx.x - 64) & 127;
    const bool issuer = tid128 == 0;
    if (grp == 0) {
      // Q row r (slot t, head g*G + r % G) into TMEM columns [TQ, TQ + 64).
      if (p.early_kv) griddep_wait();
      uint32_t w[64];
      if (valid) {
        const uint4* src = reinterpret_cast<const uint4*>(
            p.q + (((size_t)b * p.T + t) * p.Hq + g * p.G + r % p.G) * DH);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint4 u = src[i];
          w[4 * i] = u.x;
          w[4 * i + 1] = u.y;
          w[4 * i + 2] = u.z;
          w[4 * i + 3] = u.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) w[i] = 0u;
      }
      tmem_st32(tl + TQ, reinterpret_cast<const float*>(w));
      tmem_st32(tl + TQ + 32, reinterpret_cast<const float*>(w + 32));
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(q_full);
    }
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    const float c = p.scale_log2;
    const uint32_t idPV = idesc_bf16_f32(ROWS, DH, false, true);
    const uint32_t pa = smem_u32(sP) + grp * P_BYTES, va = smem_u32(sV);
    int k = 0;                                   // tiles done by this group
    for (int j = grp; j < ntiles; j += 2, ++k) {
      const int key0 = k_begin + j * BN;
      const int st = j % NST, sb = j % NSB;
      const int nv = min(BN, k_end - key0);
      bool ok_it = true;
      if (nv < BN) {
        // Zero the V rows past the sequence so that P = 0 meets finite values.
        ok_it = warp_wait(&v_full[st], (j / NST) & 1, p.status, abort_flag);
        if (ok_it) {
          uint8_t* vt = sV + st * KT_BYTES;
          const int per_half = (BN - nv) * 8;
          for (int cix = tid128; cix < 2 * per_half; cix += 128) {
            const int half = cix / per_half, rem = cix % per_half;
            const int row = nv + rem / 8;
            *reinterpret_cast<uint4*>(vt + half * 8192 + row * 128 + (rem % 8) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
      }
      if (ok_it) ok_it = warp_wait(&s_full[sb], (j / NSB) & 1, p.status, abort_flag);
      if (ok_it) {
        tc_fence_after();
        float s[BN];
        tmem_ld32(tl + TS + sb * 64, s);
        tmem_ld32(tl + TS + sb * 64 + 32, s + 32);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&s_free[sb]);
        const int lim = vis_end - key0;
        if (lim < BN) {
#pragma unroll
          for (int i = 0; i < BN; ++i) s[i] = (i < lim) ? s[i] : -INFINITY;
        }
        // row maximum of the raw scores (tree), then in scaled log2 units
        float mx[BN / 2];
#pragma unroll
        for (int i = 0; i < BN / 2; ++i) mx[i] = fmaxf(s[2 * i], s[2 * i + 1]);
#pragma unroll
        for (int w2 = BN / 4; w2 >= 1; w2 >>= 1) {
#pragma unroll
          for (int i = 0; i < w2; ++i) mx[i] = fmaxf(mx[i], mx[i + w2]);
        }
        const float mt = mx[0] * c;
        // Raise the running maximum only when it grew by more than 2^8; the
        // decision is per row, the O rescale in TMEM is warp-collective.
        float alpha = 1.f;
        const bool grow = mt > m_run + RESCALE_THRESHOLD;
        if (grow) alpha = (m_run == -INFINITY) ? 0.f : ex2(m_run - mt);
        // P buffer and O of this group are free once its previous PV completed.
        if (k > 0) ok_it = warp_wait(&o_done[grp], (k - 1) & 1, p.status, abort_flag);
        if (ok_it) {
          const bool grow_o = grow && k > 0 && m_run != -INFINITY;
          if (__any_sync(0xffffffffu, grow_o)) {
            tc_fence_after();
            const float a_o = grow_o ? alpha : 1.f;
#pragma unroll 1
            for (int cc = 0; cc < DH / 32; ++cc) {
              float o[32];
              tmem_ld32(tO + cc * 32, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] *= a_o;
              tmem_st32(tO + cc * 32, o);
            }
            tmem_wait_st();
          }
          if (grow) {
            l_run *= alpha;
            m_run = mt;
          }
          uint8_t* prow = sP + grp * P_BYTES + r * 128;
          const bool none = (m_run == -INFINITY);
          const float nm = none ? 0.f : -m_run;
          float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
          for (int cc = 0; cc < BN / 8; ++cc) {
            uint32_t wds[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float x0 = none ? 0.f : ex2(fmaf(s[cc * 8 + 2 * e], c, nm));
              const float x1 = none ? 0.f : ex2(fmaf(s[cc * 8 + 2 * e + 1], c, nm));
              sum0 += x0;
              sum1 += x1;
              wds[e] = pack_bf16x2(x0, x1);
            }
            *reinterpret_cast<uint4*>(prow + ((cc ^ (r & 7)) << 4)) =
                make_uint4(wds[0], wds[1], wds[2], wds[3]);
          }
          l_run += sum0 + sum1;
          fence_proxy_async_smem();
          tc_fence_before();
        }
      }
      // the whole group agrees, then its first thread issues O_w += P(j) V_j
      ok = group_bar_and(2 + grp, ok_it);
      if (!ok) break;
      if (issuer) {
        if (mbar_wait(&v_full[st], (j / NST) & 1, p.status, abort_flag)) {
          tc_fence_after();
          const uint32_t vb = va + st * KT_BYTES;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint64_t ad = smem_desc_sw128(pa + kk * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(vb + kk * 16 * 128, 8192, 1024);
            umma_f16(tmem + grp * DH, ad, bd, idPV, (k > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&o_done[grp]);
          umma_commit(&kv_empty[st]);
        }
      }
    }
    if (issuer) {
      // every PV this group issued has finished before TMEM is released
      umma_commit(&g_done[grp]);
      mbar_drain(&g_done[grp], 0);
    }
    // ---------------------------------------------------------- epilogue
    // both groups wait for their last PV, then merge (m, l, O) per row
    ok = __all_sync(0xffffffffu, ok);
    if (ok && k > 0) ok = warp_wait(&o_done[grp], (k - 1) & 1, p.status, abort_flag);
    // after this barrier both groups' last PV has completed: the P buffers,
    // which hold the (m, l) exchange, are free
    ok = softmax_bar_and(ok);
    if (ok) ml[grp * ROWS + r] = make_float2(m_run, l_run);
    ok = softmax_bar_and(ok);
    if (ok) {
      tc_fence_after();
      const bool has1 = ntiles > 1;
      const float2 z0 = ml[r];
      const float2 z1 = has1 ? ml[ROWS + r] : make_float2(-INFINITY, 0.f);
      const float M = fmaxf(z0.x, z1.x);
      const float w0 = (z0.x == -INFINITY) ? 0.f : ex2(z0.x - M);
      const float w1 = (z1.x == -INFINITY) ? 0.f : ex2(z1.x - M);
      const float L = w0 * z0.y + w1 * z1.y;
      const int hh = valid ? r % p.G : 0;
      const size_t unit = ((size_t)(b * p.Hkv + g) * p.nsplit_max + s_idx) * ROWS + r;
      const float inv_l = (L > 0.f) ? 1.f / L : 0.f;
      // group w writes output columns [64 w, 64 w + 64)
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        const int col = grp * 64 + cc * 32;
        float a[32], bb[32];
        tmem_ld32(tl + col, a);
        if (has1) tmem_ld32(tl + DH + col, bb);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) a[i] = w0 * a[i] + (has1 ? w1 * bb[i] : 0.f);
        if (!valid) continue;
        if (nsplit_b == 1) {
          __nv_bfloat16* dst =
              p.out + (((size_t)b * p.T + t) * p.Hq + g * p.G + hh) * DH + col;
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 v;
            v.x = pack_bf16x2(a[i] * inv_l, a[i + 1] * inv_l);
            v.y = pack_bf16x2(a[i + 2] * inv_l, a[i + 3] * inv_l);
            v.z = pack_bf16x2(a[i + 4] * inv_l, a[i + 5] * inv_l);
            v.w = pack_bf16x2(a[i + 6] * inv_l, a[i + 7] * inv_l);
            *reinterpret_cast<uint4*>(dst + i) = v;
          }
        } else {
          float* dst = p.ws_o + unit * DH + col;
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(dst + i) = make_float4(a[i], a[i + 1], a[i + 2], a[i + 3]);
        }
      }
      if (valid && nsplit_b > 1 && grp == 0) p.ws_ml[unit] = make_float2(M, L);
    }
  }

  // Each warp reconverges (warps 0 and 1 ran their roles on one lane) before
  // the CTA barrier that orders every TMEM access before the release.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Merges the KV splits of each (b, g) row: O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
// One warp per row. The splits' (m, l) are read one split per lane (32 at a
// time) and M is a warp maximum; the partial O rows (512 B, 16 B a lane) are
// added in split order, the weight and l of split s coming from lane s % 32 by
// shuffle. With at most 32 splits, every (m, l) and the first 16 partial rows
// are loaded in one round before M is known (the merge follows a kernel
// boundary, where each dependent round of loads costs about a microsecond),
// later rows eight at a time. The additions are those of a plain loop over
// s = 0, 1, ...; the batching only keeps many loads in flight.
__global__ void __launch_bounds__(128)
    attn_combine_kernel(const Params p) {
  const int g = blockIdx.y, b = blockIdx.z;
  const int r = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  griddep_launch();
  griddep_wait();
  if (r >= p.G * p.T) return;
  const int P = checked_prefix(p.kv_len[b], p.Lmax - p.T, nullptr);  // reported by the main kernel
  const int nkeys = P + p.T;
  const int ns = (nkeys + p.split - 1) / p.split;
  if (ns <= 1) return;  // written directly by the main kernel
  const size_t base = (size_t)(b * p.Hkv + g) * p.nsplit_max;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = 0.f;
  if (ns <= 32) {
    // one round of loads: every (m, l) and the first 16 splits' partial rows
    // go out together; the max and the weights follow from registers
    const float2 ml = lane < ns ? p.ws_ml[(base + lane) * ROWS + r] : make_float2(-INFINITY, 0.f);
    float4 o[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      o[j] = j < ns ? *reinterpret_cast<const float4*>(p.ws_o + ((base + j) * ROWS + r) * DH + lane * 4)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
    float M = ml.x;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float wl = (ml.x == -INFINITY) ? 0.f : ex2(ml.x - M);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float w = __shfl_sync(0xffffffffu, wl, j);
      const float l = __shfl_sync(0xffffffffu, ml.y, j);
      if (j < ns) {
        L += w * l;
        acc.x += w * o[j].x;
        acc.y += w * o[j].y;
        acc.z += w * o[j].z;
        acc.w += w * o[j].w;
      }
    }
    for (int j0 = 16; j0 < ns; j0 += 8) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        o[j] = (j0 + j < ns) ? *reinterpret_cast<const float4*>(
                                   p.ws_o + ((base + j0 + j) * ROWS + r) * DH + lane * 4)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float w = __shfl_sync(0xffffffffu, wl, (j0 + j) & 31);
        const float l = __shfl_sync(0xffffffffu, ml.y, (j0 + j) & 31);
        if (j0 + j < ns) {
          L += w * l;
          acc.x += w * o[j].x;
          acc.y += w * o[j].y;
          acc.z += w * o[j].z;
          acc.w += w * o[j].w;
        }
      }
    }
  }
  float M = -INFINITY;
  if (ns > 32) {
    for (int s0 = 0; s0 < ns; s0 += 32)
      if (s0 + lane < ns) M = fmaxf(M, p.ws_ml[(base + s0 + lane) * ROWS + r].x);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  }
  for (int s0 = 0; ns > 32 && s0 < ns; s0 += 32) {
    const int cnt = min(32, ns - s0);
    const float2 ml = lane < cnt ? p.ws_ml[(base + s0 + lane) * ROWS + r] : make_float2(-INFINITY, 0.f);
    const float wl = (ml.x == -INFINITY) ? 0.f : ex2(ml.x - M);
    for (int j0 = 0; j0 < cnt; j0 += 8) {
      float4 o[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        o[j] = (j0 + j < cnt) ? *reinterpret_cast<const float4*>(
                                    p.ws_o + ((base + s0 + j0 + j) * ROWS + r) * DH + lane * 4)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float w = __shfl_sync(0xffffffffu, wl, (j0 + j) & 31);
        const float l = __shfl_sync(0xffffffffu, ml.y, (j0 + j) & 31);
        if (j0 + j < cnt) {
          L += w * l;
          acc.x += w * o[j].x;
          acc.y += w * o[j].y;
          acc.z += w * o[j].z;
          acc.w += w * o[j].w;
        }
      }
    }
  }
  const float inv = 1.f / L;
  const int t = r / p.G, hh = r % p.G;
  __nv_bfloat16* dst = p.out + (((size_t)b * p.T + t) * p.Hq + g * p.G + hh) * DH + lane * 4;
  float d0, d1;
  uint2 v;
  v.x = pack_bf16(acc.x * inv, acc.y * inv, d0, d1);
  v.y = pack_bf16(acc.z * inv, acc.w * inv, d0, d1);
  *reinterpret_cast<uint2*>(dst) = v;
}

// Launch order of the (sequence, KV split) items of a batch with ragged
// prefixes: longest first. One CTA runs per SM and the hardware hands out
// CTAs in grid order, so this is list scheduling; taking the longest items
// first keeps a long item from starting last and leaving the other SMs idle
// (the longest-processing-time rule). A counting sort on the item's number of
// 64-key tiles: count, scan from the longest bucket down, scatter. The order
// inside a bucket is whatever the atomics give; it changes no result, since
// every item writes its own output and the merge reads the splits in split
// order.
constexpr int PLAN_THREADS = 1024;
constexpr int PLAN_BUCKETS = 4096;

__device__ __forceinline__ int plan_key(const int32_t* kv_len, int it, int T, int Lmax, int split,
                                        int nsplit, int nb) {
  const int b = it / nsplit, s = it % nsplit;
  const int P = checked_prefix(kv_len[b], Lmax - T, nullptr);  // reported by the attention kernel
  int len = P + T - s * split;
  if (len <= 0) return 0;
  len = len < split ? len : split;
  const int t = (len + BN - 1) / BN;
  return t < nb - 1 ? t : nb - 1;
}

__global__ void __launch_bounds__(PLAN_THREADS)
    attn_plan_kernel(const int32_t* __restrict__ kv_len, int B, int T, int Lmax, int split,
                     int nsplit, int32_t* __restrict__ order) {
  __shared__ int cnt[PLAN_BUCKETS];
  __shared__ int warp_sum[PLAN_THREADS / 32];
  griddep_launch();
  griddep_wait();
  const int tid = threadIdx.x;
  const int nb = min(split / BN + 1, PLAN_BUCKETS);
  for (int i = tid; i < PLAN_BUCKETS; i += PLAN_THREADS) cnt[i] = 0;
  __syncthreads();
  const int n = B * nsplit;
  for (int it = tid; it < n; it += PLAN_THREADS)
    atomicAdd(&cnt[plan_key(kv_len, it, T, Lmax, split, nsplit, nb)], 1);
  __syncthreads();
  // Exclusive scan over the buckets from the longest (nb - 1) down to 0:
  // thread j owns reversed positions 4j .. 4j+3.
  constexpr int PER = PLAN_BUCKETS / PLAN_THREADS;
  int c[PER], local = 0;
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int r = tid * PER + k;
    c[k] = r < nb ? cnt[nb - 1 - r] : 0;
    local += c[k];
  }
  const int lane = tid & 31, w = tid >> 5;
  int incl = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) warp_sum[w] = incl;
  __syncthreads();
  if (w == 0) {
    int x = warp_sum[lane], xi = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, xi, off);
      if (lane >= off) xi += y;
    }
    warp_sum[lane] = xi - x;  // exclusive prefix of the warp totals
  }
  __syncthreads();
  int start = warp_sum[w] + incl - local;
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int r = tid * PER + k;
    if (r < nb) cnt[nb - 1 - r] = start;
    start += c[k];
  }
  __syncthreads();
  for (int it = tid; it < n; it += PLAN_THREADS) {
    const int pos = atomicAdd(&cnt[plan_key(kv_len, it, T, Lmax, split, nsplit, nb)], 1);
    order[pos] = it;
  }
}

}  // namespace attn

// KV split length (keys per CTA) for a launch of B x Hkv sequences of at most
// Lmax keys. One CTA runs per SM, so the time is about
//   ceil(CTAs / SMs) * (tiles per split + per-CTA overhead) + merge,
// where the per-CTA overhead (start-up, first loads, partial write and the
// tail of a wave) is worth about forty 64-key tiles and the merge launch,
// when the keys are split, about eight (calibrated on B300 by sweeping the
// split length of the batch-1/4096, batch-4/32768 and batch-64 workloads).
// The smallest cost wins; ties keep the longer split.
int attn_bf16_auto_split(int B, int Hkv, int Lmax) {
  const long long sms = num_sms();
  const long long tiles = (Lmax + attn::BN - 1) / attn::BN;
  long long best = -1;
  int best_split = (int)(tiles * attn::BN);
  for (long long per = tiles; per >= 1; --per) {
    const long long nsplit = (tiles + per - 1) / per;
    if (per > 1 && (tiles + per - 2) / (per - 1) == nsplit) continue;  // same split count, shorter
    const long long ctas = (long long)B * Hkv * nsplit;
    const long long waves = (ctas + sms - 1) / sms;
    const long long cost = waves * (per + 40) + (nsplit > 1 ? 8 : 0);
    if (best < 0 || cost < best) {
      best = cost;
      best_split = (int)(per * attn::BN);
    }
    if (nsplit >= 256) break;
  }
  return best_split;
}

// Workspace: the per-split partial results when the keys are split, then,
// for a batch of more than one sequence, the launch order of its items.
static size_t attn_partials_bytes(int B, int Hkv, int nsplit) {
  if (nsplit <= 1) return 0;
  return (size_t)B * Hkv * nsplit * attn::ROWS * (attn::DH * sizeof(float) + sizeof(float2));
}

static size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

size_t attn_bf16_workspace(int B, int T, int Hq, int Hkv, int Lmax, int split) {
  (void)T;
  (void)Hq;
  const int nsplit = (Lmax + split - 1) / split;
  size_t bytes = attn_partials_bytes(B, Hkv, nsplit);
  if (B > 1) bytes = round256(bytes) + round256((size_t)B * nsplit * sizeof(int32_t));
  return bytes;
}

ndiff_status launch_attn_bf16(const void* q, const void* k, const void* v, const int32_t* kv_len,
                              int B, int T, int Hq, int Hkv, int Lmax, int causal, float scale,
                              int split, void* out, void* ws, size_t ws_bytes,
                              cudaStream_t stream, const int4* remap, int ncache, int early_kv,
                              const void* l2pf, size_t l2pf_bytes, const void* rpf, int rpf_U,
                              int rpf_G) {
  const int G = Hq / Hkv;
  const int nsplit = (Lmax + split - 1) / split;
  const size_t need = attn_bf16_workspace(B, T, Hq, Hkv, Lmax, split);
  if (need > 0 && (ws == nullptr || ws_bytes < need))
    return set_error(NDIFF_ERR_WORKSPACE, "ndiff_block_attn: workspace of %zu bytes needed, %zu given",
                     need, ws_bytes);
  CUtensorMap tk, tv;
  {
    // the caches the launch reads: B of them, or ncache when sequences share
    // caches through the remap table
    const uint64_t dims[2] = {128, (uint64_t)(remap != nullptr ? ncache : B) * Hkv * Lmax};
    const uint64_t strides[1] = {128 * 2};
    const uint32_t box[2] = {64, (uint32_t)attn::BN};
    ndiff_status s = make_tmap_bf16(&tk, k, 2, dims, strides, box);
    if (s != NDIFF_OK) return s;
    s = make_tmap_bf16(&tv, v, 2, dims, strides, box);
    if (s != NDIFF_OK) return s;
  }
  attn::Params prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.kv_len = kv_len;
  prm.B = B;
  prm.T = T;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.G = G;
  prm.Lmax = Lmax;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.causal = causal;
  prm.split = split;
  prm.nsplit_max = nsplit;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.kc = static_cast<const __nv_bfloat16*>(k);
  prm.vc = static_cast<const __nv_bfloat16*>(v);
  prm.remap = remap;
  prm.ncache = remap != nullptr ? ncache : B;
  // early K/V needs a final kv_len and no table written by the launch before
  // (no remap, no launch order: one sequence)
  prm.early_kv = (early_kv && remap == nullptr && B == 1) ? 1 : 0;
  // the prefetch wants 16-byte aligned addresses and sizes
  const bool pf_ok = l2pf != nullptr && (reinterpret_cast<uintptr_t>(l2pf) & 15) == 0;
  prm.l2pf = pf_ok ? static_cast<const char*>(l2pf) : nullptr;
  prm.l2pf_bytes = pf_ok ? (l2pf_bytes & ~(size_t)15) : 0;
  const bool rpf_ok = pf_ok && rpf != nullptr && (reinterpret_cast<uintptr_t>(rpf) & 15) == 0 && rpf_G > 0 &&
                      rpf_U > 0;
  prm.rpf = rpf_ok ? static_cast<const char*>(rpf) : nullptr;
  prm.rpf_U = rpf_ok ? rpf_U : 0;
  prm.rpf_G = rpf_ok ? rpf_G : 1;
  prm.ws_o = static_cast<float*>(ws);
  const size_t partials = attn_partials_bytes(B, Hkv, nsplit);
  prm.ws_ml = partials ? reinterpret_cast<float2*>(static_cast<uint8_t*>(ws) +
                                                   (size_t)B * Hkv * nsplit * attn::ROWS *
                                                       attn::DH * sizeof(float))
                       : nullptr;
  int32_t* order = B > 1 ? reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + round256(partials))
                         : nullptr;
  prm.order = order;
  prm.status = device_status_word();
  static bool attr_set[64] = {false};
  int dev = 0;
  NDIFF_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 64 && !attr_set[dev]) {
    NDIFF_CUDA_TRY(cudaFuncSetAttribute(attn::attn_bf16_kernel,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        attn::SMEM_BYTES));
    attr_set[dev] = true;
  }
  dim3 grid(nsplit, Hkv, B);
  if (order != nullptr) {
    NDIFF_CUDA_TRY(launch_k(attn::attn_plan_kernel, dim3(1), dim3(attn::PLAN_THREADS), 0, stream,
                            kv_len, B, T, Lmax, split, nsplit, order));
    grid = dim3(nsplit * Hkv * B, 1, 1);
  }
  NDIFF_CUDA_TRY(launch_k(attn::attn_bf16_kernel, grid, dim3(attn::THREADS),
                          (size_t)attn::SMEM_BYTES, stream, tk, tv, prm));
  if (nsplit > 1) {
    dim3 g2((G * T + 3) / 4, Hkv, B);
    NDIFF_CUDA_TRY(launch_k(attn::attn_combine_kernel, g2, dim3(128), 0, stream, prm));
  }
  return NDIFF_OK;
}

}  // namespace ndiff
