// gemm_wide.cu — the model's projections for a batch of sequences on sm_103a:
// y[m][n] = sum_k x[m][k] W[n][k] for any number M of token rows (B sequences
// of T tokens, M = B*T) against a bf16 weight matrix W [N][K].
//
// Where it sits: the same linear maps as gemm_bf16.cu (QKV, output projection,
// SwiGLU gate/up, down projection, LM head), run for many sequences at once,
// which is how a server decodes at high concurrency ("Nemotron-Labs-Diffusion:
// A Tri-Mode Language Model ..." (hotpaper.ai), Abstract: the modes are chosen
// to sustain throughput across deployment settings and concurrency levels).
// At B = 64 block forwards (2048 token rows) the work is 2 * 2048 flops per
// weight byte pair: tensor-bound, so each weight tile is used for 256 token
// columns per MMA and the token chunks of one tile run back to back.
//
// Design (swap-AB as in the skinny kernel: the weight tile is the 128-row A
// operand, 256 token rows are the MMA's N = 256 columns, so an accumulator is
// 128 lanes x 256 fp32 columns of TMEM; two accumulators fill the 512 columns):
//   * Work items are (128-row tile of W, 256-row chunk of tokens), tile-major,
//     so the chunks of one weight tile are taken by neighbouring CTAs at about
//     the same time and all but the first read the tile from L2. A persistent
//     grid of at most one CTA per SM walks the items round-robin.
//   * Warp 0 streams 128x64 weight tiles and 256x64 activation tiles through a
//     4-stage TMA ring (48 KB a stage, 128-byte swizzle); warp 1 issues
//     tcgen05.mma M128 N256 K16; warps 2-5 drain the other accumulator in
//     32-column slices, so the epilogue of one item overlaps the next item's
//     main loop. Launches of at most 64 rows (a batch's AR step) use 64-row
//     chunks (M128 N64) and an 8-stage ring of 24 KB. No K split in either, so
//     a row's arithmetic is the same in AR and block forwards.
//   * Fused epilogues as in the skinny kernel, for token rows of several
//     sequences: fp32 store, residual add, SwiGLU, QKV with RoPE and the K/V
//     write at each token's own sequence and position, and the ARGMAX
//     reduction of the LM head (per 128-id tile and token row).
//   * Every mbarrier wait is bounded; on expiry the kernel records a timeout in
//     the device status word, lets issued TMA copies land, frees TMEM and exits.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace ndiff {
namespace gemm_wide {

constexpr int BM = 128;                     // weight rows per tile (MMA M)
constexpr int BK = 64;                      // K per stage (one 128-byte swizzle atom)
constexpr int A_BYTES = BM * BK * 2;        // 16 KB
constexpr int THREADS = 192;
constexpr float L2E = 1.4426950408889634f;

// Geometry for MT token rows per item (the MMA's N): 256 for block forwards
// of a batch (4 stages of 48 KB), 64 for the AR forward of up to 64
// sequences (8 stages of 24 KB: twice the weight bytes in flight per SM, for
// the short projections that have fewer weight tiles than SMs). Both run the
// same K loop with no split, so a row's arithmetic is the same in either.
template <int MT_>
struct Geo {
  static constexpr int MT = MT_;
  static constexpr int NST = MT_ == 256 ? 4 : 8;
  static constexpr int B_BYTES = MT_ * BK * 2;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + NST * A_BYTES;
  static constexpr int OFF_RED = OFF_B + NST * B_BYTES;  // ARGMAX: [4 warps][32 tokens] float4
  static constexpr int RED_BYTES = 4 * 32 * 16;
  static constexpr int OFF_BAR = OFF_RED + RED_BYTES;
  static constexpr int N_BARS = 2 * NST + 4 + 1;
  static constexpr int SMEM_BYTES = OFF_BAR + N_BARS * 8 + 64 + 1024;
  static constexpr int TMEM_COLS = 2 * MT_;             // two accumulators
};

static_assert(Geo<256>::OFF_B % 1024 == 0 && Geo<64>::OFF_B % 1024 == 0,
              "swizzled tiles need 1024-byte alignment");
static_assert(Geo<256>::SMEM_BYTES <= 227 * 1024 && Geo<64>::SMEM_BYTES <= 227 * 1024,
              "shared memory per CTA");

__device__ __forceinline__ void bar_sync128() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ bool bar_and(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t b = smem_u32(bar);
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(b, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) return;
  }
}

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------- epilogues
// Thread r holds y[storage row tile*128 + r][token m0 + j] in v[j], j < 32.
__device__ __forceinline__ void epilogue(const GemmParams& p, int tile, int r, int m0,
                                         const float (&v)[32]) {
  const int n = tile * BM + r;
  switch (p.mode) {
    case GEMM_EPI_F32: {
      if (n < p.N) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (m0 + j < p.T) p.out[(size_t)(m0 + j) * p.ldo + n] = v[j];
      }
      break;
    }
    case GEMM_EPI_RESID: {
      if (n < p.N) {
        float old[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) old[j] = (m0 + j < p.T) ? p.out[(size_t)(m0 + j) * p.ldo + n] : 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (m0 + j < p.T) p.out[(size_t)(m0 + j) * p.ldo + n] = old[j] + v[j];
      }
      break;
    }
    case GEMM_EPI_SWIGLU: {
      // even rows: gate j = tile*64 + r/2; odd rows: up of the same j
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float u = __shfl_xor_sync(0xffffffffu, v[j], 1);
        if (!(r & 1) && m0 + j < p.T) {
          const float g = v[j];
          p.act[(size_t)(m0 + j) * p.lda + tile * 64 + (r >> 1)] =
              __float2bfloat16_rn(g / (1.f + expf(-g)) * u);
        }
      }
      break;
    }
    case GEMM_EPI_QKV: {
      // Tile = one head (q heads, then k heads, then v heads). Token m is slot
      // m % Tb of sequence m / Tb, at position kv_len[b] + slot.
      const int h = tile;
      const bool rot = h < p.Hq + p.Hkv;
      const int i = r >> 1;
      const int dim = rot ? ((r & 1) ? i + 64 : i) : r;
      float pv[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) pv[j] = __shfl_xor_sync(0xffffffffu, v[j], 1);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int m = m0 + j;
        if (m >= p.T) continue;
        const int b = m / p.Tb, slot = m - b * p.Tb;
        const int P = checked_prefix(__ldg(p.kv_len + b), p.Lmax - p.Tb, p.status);
        const int pos = P + slot;
        float y = v[j];
        if (rot) {
          const float2 cs = __ldg(p.rope + (size_t)pos * 64 + i);
          y = (r & 1) ? y * cs.x + pv[j] * cs.y : y * cs.x - pv[j] * cs.y;
        }
        __nv_bfloat16* dst;
        if (h < p.Hq)
          dst = p.q + ((size_t)m * p.Hq + h) * BM + dim;
        else if (h < p.Hq + p.Hkv)
          dst = p.kc + (((size_t)b * p.Hkv + (h - p.Hq)) * p.Lmax + pos) * BM + dim;
        else
          dst = p.vc + (((size_t)b * p.Hkv + (h - p.Hq - p.Hkv)) * p.Lmax + pos) * BM + dim;
        *dst = __float2bfloat16_rn(y);
      }
      break;
    }
    default:
      break;
  }
}

// ARGMAX: the LM-head tile's per-token softmax state and best allowed id, as in
// the skinny kernel (lane-halving transpose-reduction inside each warp, the
// four warps merged in order through shared memory); the tile's states go to
// red[tile][m] (row stride M).
struct Red {
  float m, s, bv;
  int bi;
};

__device__ __forceinline__ void red_merge(Red& a, const Red& b) {
  if (b.m > a.m) {
    a.s = b.s + (a.m == -INFINITY ? 0.f : a.s * ex2f((a.m - b.m) * L2E));
    a.m = b.m;
  } else {
    a.s += (b.m == -INFINITY ? 0.f : b.s * ex2f((b.m - a.m) * L2E));
  }
  if (b.bv > a.bv || (b.bv == a.bv && b.bi < a.bi)) {
    a.bv = b.bv;
    a.bi = b.bi;
  }
}

__device__ __forceinline__ Red red_shfl(const Red& a, int off) {
  Red o;
  o.m = __shfl_xor_sync(0xffffffffu, a.m, off);
  o.s = __shfl_xor_sync(0xffffffffu, a.s, off);
  o.bv = __shfl_xor_sync(0xffffffffu, a.bv, off);
  o.bi = __shfl_xor_sync(0xffffffffu, a.bi, off);
  return o;
}

template <int W>
__device__ __forceinline__ void red_halve(Red (&a)[W], Red (&o)[W / 2], int lane, int off) {
  const bool hi = (lane & off) != 0;
#pragma unroll
  for (int j = 0; j < W / 2; ++j) {
    Red keep = hi ? a[j + W / 2] : a[j];
    const Red send = hi ? a[j] : a[j + W / 2];
    red_merge(keep, red_shfl(send, off));
    o[j] = keep;
  }
}

__device__ __forceinline__ void epilogue_argmax(const GemmParams& p, int tile, int r, int lane,
                                                int quarter, int m0, const float (&v)[32],
                                                float4* sred) {
  const int n = tile * BM + r;
  const bool valid = n < p.N;
  const bool allowed = valid && n != p.excl;
  Red a16[16];
  {
    const bool hi = (lane & 16) != 0;
    const int n2 = n ^ 16;
    const bool valid2 = n2 < p.N, allowed2 = valid2 && n2 != p.excl;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float keep = hi ? v[j + 16] : v[j];
      const float send = hi ? v[j] : v[j + 16];
      const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
      const float x0 = valid ? keep : -INFINITY;
      const float x1 = valid2 ? recv : -INFINITY;
      Red t;
      t.m = fmaxf(x0, x1);
      t.s = (t.m == -INFINITY) ? 0.f
                               : ((x0 == -INFINITY ? 0.f : ex2f((x0 - t.m) * L2E)) +
                                  (x1 == -INFINITY ? 0.f : ex2f((x1 - t.m) * L2E)));
      const float b0 = allowed ? keep : -INFINITY, b1 = allowed2 ? recv : -INFINITY;
      const int i0 = allowed ? n : 0x7fffffff, i1 = allowed2 ? n2 : 0x7fffffff;
      const bool take1 = b1 > b0 || (b1 == b0 && i1 < i0);
      t.bv = take1 ? b1 : b0;
      t.bi = take1 ? i1 : i0;
      a16[j] = t;
    }
  }
  Red a8[8], a4[4], a2[2], a1[1];
  red_halve<16>(a16, a8, lane, 8);
  red_halve<8>(a8, a4, lane, 4);
  red_halve<4>(a4, a2, lane, 2);
  red_halve<2>(a2, a1, lane, 1);
  sred[quarter * 32 + lane] = make_float4(a1[0].m, a1[0].s, a1[0].bv, __int_as_float(a1[0].bi));
  bar_sync128();
  if (quarter == 0 && m0 + lane < p.T) {
    float4 f = sred[lane];
    Red acc{f.x, f.y, f.z, __float_as_int(f.w)};
#pragma unroll
    for (int q = 1; q < 4; ++q) {
      f = sred[q * 32 + lane];
      red_merge(acc, Red{f.x, f.y, f.z, __float_as_int(f.w)});
    }
    __stcg(p.red + (size_t)tile * p.T + m0 + lane,
           make_float4(acc.m, acc.s, acc.bv, __int_as_float(acc.bi)));
  }
  bar_sync128();
}

// ---------------------------------------------------------------- kernel
template <int MT, bool ARGMAX>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_wide_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                     const GemmParams p, int nchunks) {
  using G = Geo<MT>;
  constexpr int NST = G::NST, B_BYTES = G::B_BYTES, OFF_A = G::OFF_A, OFF_B = G::OFF_B;
  constexpr int OFF_RED = G::OFF_RED, OFF_BAR = G::OFF_BAR, N_BARS = G::N_BARS;
  constexpr int TMEM_COLS = G::TMEM_COLS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem + OFF_A;
  uint8_t* sB = smem + OFF_B;
  float4* sred = reinterpret_cast<float4*>(smem + OFF_RED);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* full = bars;
  uint64_t* empty = full + NST;
  uint64_t* acc_full = empty + NST;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* mma_done = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + N_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 128);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
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
  const int grid = gridDim.x;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      griddep_wait();
      int kc = 0;
      bool ok = true;
      for (int it = blockIdx.x; ok && it < p.items; it += grid) {
        const int tile = it / nchunks, chunk = it % nchunks;
        for (int ks = 0; ks < p.nks; ++ks) {
          const int st = kc % NST;
          if (kc >= NST && !mbar_wait(&empty[st], ((kc / NST) - 1) & 1, p.status, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[st], A_BYTES + B_BYTES);
          if (p.w_tiled)
            tma_load_2d(sA + st * A_BYTES, &tmW, &full[st], 0, (tile * p.nks + ks) * BM);
          else
            tma_load_2d(sA + st * A_BYTES, &tmW, &full[st], ks * BK, tile * BM);
          tma_load_2d(sB + st * B_BYTES, &tmX, &full[st], ks * BK, chunk * MT);
          ++kc;
        }
      }
      if (*abort_flag) {
        for (int j = (kc > NST ? kc - NST : 0); j < kc; ++j) mbar_drain(&full[j % NST], (j / NST) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(BM, MT, false, false);
      const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
      int kc = 0, ic = 0;
      bool ok = true;
      for (int it = blockIdx.x; ok && it < p.items; it += grid) {
        const int buf = ic & 1;
        if (ic >= 2 && !mbar_wait(&acc_empty[buf], ((ic >> 1) - 1) & 1, p.status, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + buf * MT;
        for (int ks = 0; ks < p.nks; ++ks) {
          const int st = kc % NST;
          if (!mbar_wait(&full[st], (kc / NST) & 1, p.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = smem_desc_sw128(a0 + st * A_BYTES + kk * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(b0 + st * B_BYTES + kk * 32, 16, 1024);
            umma_f16(d, ad, bd, idesc, (ks > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&empty[st]);
          ++kc;
        }
        if (!ok) break;
        umma_commit(&acc_full[buf]);
        ++ic;
      }
      // every MMA issued above has finished before TMEM is released
      umma_commit(mma_done);
      mbar_drain(mma_done, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const uint32_t quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t tl = tmem + ((quarter * 32u) << 16);
    griddep_wait();
    int ic = 0;
    for (int it = blockIdx.x; it < p.items; it += grid, ++ic) {
      const int buf = ic & 1;
      bool ok = mbar_wait(&acc_full[buf], (ic >> 1) & 1, p.status, abort_flag);
      if (!bar_and(ok)) break;
      tc_fence_after();
      const int tile = it / nchunks, chunk = it % nchunks;
      const int ncols = min(MT, ((p.T - chunk * MT) + 31) & ~31);  // 32-column slices with tokens
#pragma unroll 1
      for (int c = 0; c < ncols; c += 32) {
        float v[32];
        tmem_ld32(tl + buf * MT + c, v);
        tmem_wait_ld();
        if constexpr (ARGMAX)
          epilogue_argmax(p, tile, r, (int)lane, (int)quarter, chunk * MT + c, v, sred);
        else
          epilogue(p, tile, r, chunk * MT + c, v);
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[buf]);
    }
  }

  __syncwarp();  // warps 0 and 1 reconverge before the CTA barrier
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace gemm_wide

static int wide_mt(int M) { return gemm_wide_box_rows(M); }

GemmPlan gemm_wide_plan(int N, int K, int M) {
  GemmPlan pl;
  const int mt = wide_mt(M);
  pl.ntiles = (N + gemm_wide::BM - 1) / gemm_wide::BM;
  pl.nks = K / gemm_wide::BK;
  pl.S = 1;
  pl.nchunks = (M + mt - 1) / mt;
  pl.items = pl.ntiles * pl.nchunks;
  const int sms = num_sms();
  pl.grid = pl.items < sms ? pl.items : sms;
  return pl;
}

ndiff_status gemm_wide_make_xmap(const void* x, int M, int K, CUtensorMap* tmX, int box_rows) {
  const uint64_t dims[2] = {(uint64_t)K, (uint64_t)M};
  const uint64_t strides[1] = {(uint64_t)K * 2};
  const uint32_t box[2] = {gemm_wide::BK, (uint32_t)box_rows};
  return make_tmap_bf16(tmX, x, 2, dims, strides, box);
}

template <int MT, bool ARGMAX>
static ndiff_status launch_wide_variant(const CUtensorMap& tmW, const CUtensorMap& tmX,
                                        const GemmPlan& pl, const GemmParams& p,
                                        cudaStream_t stream) {
  static bool attr_set[64] = {false};
  int dev = 0;
  NDIFF_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 64 && !attr_set[dev]) {
    NDIFF_CUDA_TRY(cudaFuncSetAttribute(gemm_wide::gemm_wide_kernel<MT, ARGMAX>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        gemm_wide::Geo<MT>::SMEM_BYTES));
    attr_set[dev] = true;
  }
  NDIFF_CUDA_TRY(launch_k(gemm_wide::gemm_wide_kernel<MT, ARGMAX>, dim3(pl.grid),
                          dim3(gemm_wide::THREADS), (size_t)gemm_wide::Geo<MT>::SMEM_BYTES, stream,
                          tmW, tmX, p, pl.nchunks));
  return NDIFF_OK;
}

ndiff_status launch_gemm_wide(const CUtensorMap& tmW, const CUtensorMap& tmX, const GemmPlan& pl,
                              GemmParams p, cudaStream_t stream) {
  if (p.T <= 0) return NDIFF_OK;
  p.S = 1;
  p.nks = pl.nks;
  p.items = pl.items;
  p.status = device_status_word();
  const bool am = p.mode == GEMM_EPI_ARGMAX;
  if (wide_mt(p.T) == 64)
    return am ? launch_wide_variant<64, true>(tmW, tmX, pl, p, stream)
              : launch_wide_variant<64, false>(tmW, tmX, pl, p, stream);
  return am ? launch_wide_variant<256, true>(tmW, tmX, pl, p, stream)
            : launch_wide_variant<256, false>(tmW, tmX, pl, p, stream);
}

}  // namespace ndiff
