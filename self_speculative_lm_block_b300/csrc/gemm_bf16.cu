// gemm_bf16.cu — the model's projections on sm_103a: y[m][n] = sum_k x[m][k] W[n][k]
// for a block of at most 32 token rows (the 32-token block of the decode step,
// or one token in AR mode) against a bf16 weight matrix W [N][K].
//
// Where it sits: every linear map of the pre-norm transformer (QKV, output
// projection, SwiGLU gate/up, down projection, LM head) that one checkpoint
// runs in all three decode modes ("NVIDIA 发布 Nemotron-Labs Diffusion 语言模型
// 系列" (fintech-frontier-insights), "三种生成模式"). Decode is bound by the
// bytes of the weights ("NVIDIA 发布 Nemotron-Labs Diffusion：三模态语言模型统一
// AR 与扩散解码" (aimodeling.com), on memory-I/O-bound decoding), so the kernel is
// a weight stream with the tensor cores doing 32 columns of work per weight.
//
// Design (swap-AB: the weight tile is the MMA's 128-row A operand, the token
// rows are its N = MT columns (32, or 64 / 128 for the fused and quadratic
// forwards), so the accumulator is 128 lanes x MT fp32 columns of TMEM):
//   * Stream-K: one CTA per SM; CTA c owns the contiguous run
//     [c U / G, (c + 1) U / G) of all tiles' k-steps (U = tiles x K / 64), in
//     tiled weight storage a contiguous run of 16 KB boxes. Warp 0 streams the
//     128x64 weight tiles and the matching MTx64 activation tiles through a TMA
//     ring (128-byte swizzle; the weight loads carry an L2 evict-first hint);
//     warp 1 issues tcgen05.mma (M128 N MT K16) into one of two TMEM
//     accumulators, one per segment (the part of one tile a CTA owns); warps
//     2-5 drain the other accumulator, so the epilogue of one segment overlaps
//     the loads of the next.
//   * One CTA per SM (~124 KB of shared memory at MT = 32: a six-stage ring).
//     Under programmatic dependent launch the next projection's CTAs start as
//     the running ones leave their SMs and stream their first six weight tiles
//     (which no earlier kernel writes, ~14 MB over the GPU) before
//     griddepcontrol.wait, i.e. while the small merge kernel between the two
//     projections runs; the activation tiles and every global write come after
//     it. With two CTAs per SM the next projection started next to the running
//     one, its prefetch competed with that projection's own stream, and HBM
//     sat idle during the merge kernel (8B: 3.38 vs 3.27 ms per AR forward).
//   * Segments of a tile split over several CTAs: with GEMM_EPI_PARTIAL (the
//     model's forward of one sequence) each segment stores its partial tile
//     and the kernel after the projection sums them; with the other epilogues
//     the last contributor to arrive at a per-tile counter adds the partials in
//     k order and runs the epilogue, then resets the counter. The partition
//     depends only on (N, K, grid), never on the number of token rows, so a
//     token row's result is the same whether it is computed alone (AR) or
//     inside a block.
//   * Fused epilogues: fp32 store (logits), residual add (x += y), SwiGLU and
//     QKV with rotate-half RoPE from a precomputed table plus the K/V-cache
//     write at the block's positions, the LM head's argmax (its own
//     instantiation). The weights are stored so that the two rows an epilogue
//     combines are adjacent (gate j / up j; RoPE dims i / i+64 of a q or k
//     head), i.e. held by neighbouring lanes, and one warp shuffle brings them
//     together.
//   * Every mbarrier wait is bounded; on expiry the kernel records a timeout in
//     the device status word, lets issued TMA copies land, frees TMEM and exits.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace ndiff {
namespace gemm {

constexpr int BM = 128;                    // weight rows per tile (MMA M)
constexpr int BK = 64;                     // K per stage (one 128-byte swizzle atom)
constexpr int A_BYTES = BM * BK * 2;       // 16 KB
constexpr int THREADS = 192;

// Shared-memory and TMEM geometry for MT token rows (the MMA's N): 32 for a
// block or one token, 64 for the fused verify + draft forward of two blocks,
// 128 for the quadratic forward (verification and three draft blocks).
template <int MT_>
struct Geo {
  static constexpr int MT = MT_;
  static constexpr int NST = MT_ == 32 ? 6 : (MT_ == 64 ? 7 : 6);  // pipeline stages
  static constexpr int B_BYTES = MT_ * BK * 2;           // 4 KB / 8 KB
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + NST * A_BYTES;
  static constexpr int OFF_RED = OFF_B + NST * B_BYTES;  // ARGMAX: [4 warps][32 tokens] float4
  static constexpr int RED_BYTES = 4 * 32 * 16;
  static constexpr int OFF_BAR = OFF_RED + RED_BYTES;
  static constexpr int N_BARS = 2 * NST + 4 + 1;
  static constexpr int SMEM_BYTES = OFF_BAR + N_BARS * 8 + 64 + 1024;
  static constexpr int TMEM_COLS = 2 * MT_;              // two accumulators
  static constexpr int MIN_BLOCKS = 1;
};

static_assert(Geo<32>::OFF_B % 1024 == 0 && Geo<64>::OFF_B % 1024 == 0,
              "swizzled tiles need 1024-byte alignment");
// At 32 token rows six stages take ~124 KB, so one CTA runs per SM (see the
// file header for why that is faster than two).
static_assert(Geo<32>::SMEM_BYTES <= 227 * 1024 && 2 * Geo<32>::SMEM_BYTES > 228 * 1024,
              "one CTA per SM at 32 token rows");
static_assert(Geo<64>::SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
static_assert(Geo<128>::OFF_B % 1024 == 0 && Geo<128>::SMEM_BYTES <= 227 * 1024,
              "shared memory per CTA at 128 token rows");

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

__device__ __forceinline__ void bar_sync128() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t b = smem_u32(bar);
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(b, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) return;
  }
}


// Epilogue of one finished 128-row tile. Thread r holds y[m0 + j] for storage
// row tile*128 + r and token rows m0 + j < T (j < W). Loads are issued before
// stores so that the token rows do not serialise on memory latency.
// QKV rows: token row m has RoPE position pos(m) and cache row slot(m): both
// kv_len[0] + m, or, with blk_pos, blk_pos[2b] + m % 32 and blk_pos[2b + 1] +
// m % 32 for its 32-row block b (the draft blocks of the quadratic forward
// sit at other positions and cache rows than the block under verification).
template <int W>
__device__ __forceinline__ void epilogue(const GemmParams& p, int tile, int r, float (&v)[W], int m0) {
  const int n = tile * BM + r;
  switch (p.mode) {
    case GEMM_EPI_F32: {
      if (n < p.N) {
#pragma unroll
        for (int j = 0; j < W; ++j)
          if (m0 + j < p.T) p.out[(size_t)(m0 + j) * p.ldo + n] = v[j];
      }
      break;
    }
    case GEMM_EPI_RESID: {
      if (n < p.N) {
        float old[W];
#pragma unroll
        for (int j = 0; j < W; ++j) old[j] = (m0 + j < p.T) ? p.out[(size_t)(m0 + j) * p.ldo + n] : 0.f;
#pragma unroll
        for (int j = 0; j < W; ++j)
          if (m0 + j < p.T) p.out[(size_t)(m0 + j) * p.ldo + n] = old[j] + v[j];
      }
      break;
    }
    case GEMM_EPI_SWIGLU: {
      // even rows: gate j = tile*64 + r/2; odd rows: up of the same j
#pragma unroll
      for (int j = 0; j < W; ++j) {
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
      // tile = one head: q heads, then k heads, then v heads. In q and k heads
      // even rows hold dim i = r/2 and odd rows dim i + 64 (the RoPE pair).
      const int P = checked_prefix(p.kv_len[0], p.Lmax - p.T, p.status);
      const int h = tile;
      const bool rot = h < p.Hq + p.Hkv;
      const int i = r >> 1;
      const int dim = rot ? ((r & 1) ? i + 64 : i) : r;
      float pv[W];
#pragma unroll
      for (int j = 0; j < W; ++j) pv[j] = __shfl_xor_sync(0xffffffffu, v[j], 1);
      const bool isq = h < p.Hq;
      __nv_bfloat16* base;
      if (isq)
        base = p.q + (size_t)h * BM + dim;
      else if (h < p.Hq + p.Hkv)
        base = p.kc + (size_t)(h - p.Hq) * p.Lmax * BM + dim;
      else
        base = p.vc + (size_t)(h - p.Hq - p.Hkv) * p.Lmax * BM + dim;
#pragma unroll
      for (int j0 = 0; j0 < W; j0 += 8) {
        int pos[8], slot[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int m = m0 + j0 + j;
          if (p.blk_pos != nullptr) {
            pos[j] = p.blk_pos[2 * (m >> 5)] + (m & 31);
            slot[j] = p.blk_pos[2 * (m >> 5) + 1] + (m & 31);
          } else {
            pos[j] = P + m;
            slot[j] = P + m;
          }
        }
        float2 cs[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          cs[j] = (rot && m0 + j0 + j < p.T) ? __ldg(p.rope + (size_t)pos[j] * 64 + i)
                                             : make_float2(1.f, 0.f);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int m = m0 + j0 + j;
          if (m < p.T) {
            float y = v[j0 + j];
            if (rot)
              y = (r & 1) ? y * cs[j].x + pv[j0 + j] * cs[j].y : y * cs[j].x - pv[j0 + j] * cs[j].y;
            const size_t at = isq ? (size_t)m * p.Hq * BM : (size_t)slot[j] * BM;
            base[at] = __float2bfloat16_rn(y);
          }
        }
      }
      break;
    }
    default:
      break;
  }
}

// ---------------------------------------------------------------- ARGMAX
// The LM head with the greedy decision fused in: instead of storing logits,
// each finished 128-row vocabulary tile leaves, per token row, the running
// softmax state (max m, sum of exp(y - m)) and the best allowed (value, id),
// ties to the lower id. A second kernel merges the tiles in tile order.
constexpr float L2E = 1.4426950408889634f;

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

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

// One halving step of the warp transpose-reduction: the lane keeps the half
// of its W columns selected by its `off` bit and merges in the partner's copy
// of that half.
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

// Thread r of the epilogue holds y[vocab n = tile*128 + r][token m] in v[m].
// Token columns m0 .. m0+31 of the tile; the states go to red[tile * stride + m].
__device__ __forceinline__ void epilogue_argmax(const GemmParams& p, int tile, int r, int lane,
                                                int quarter, const float* v, float4* sred,
                                                int stride, int m0) {
  const int n = tile * BM + r;
  const bool valid = n < p.N;
  const bool allowed = valid && n != p.excl;
  // step 1 (offset 16) starts from single elements
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
  // lane l now holds token column l over this warp's 32 vocabulary rows
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
    __stcg(p.red + (size_t)tile * stride + m0 + lane,
           make_float4(acc.m, acc.s, acc.bv, __int_as_float(acc.bi)));
  }
  bar_sync128();
}

// ARGMAX selects the LM-head epilogue at compile time: a separate
// instantiation keeps that epilogue's registers and code out of the
// projections' kernel (measured 7% slower decode when both shared one body).
template <int MT, bool ARGMAX>
__global__ void __launch_bounds__(THREADS, Geo<MT>::MIN_BLOCKS)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                     const GemmParams p) {
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
  volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);

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
    *last_flag = 0;
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
  // stream-K partition: CTA c owns k-steps [c U / G, (c + 1) U / G) of the
  // U = ntiles * nks k-steps; it depends on (N, K, grid) only, never on the
  // token rows, so a row's arithmetic is the same in every launch
  // (32-bit arithmetic: the launcher keeps U * (grid + 1) below 2^31)
  const int U = p.ntiles * p.nks;
  const int kb0 = (int)((long long)blockIdx.x * U / gridDim.x);
  const int kb1 = (int)((long long)(blockIdx.x + 1) * U / gridDim.x);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      // This CTA's k-steps are the contiguous run [kb0, kb1) of all tiles' k-steps
      // (k-step g is k-step g % nks of tile g / nks; in tiled storage it is the
      // 16 KB run of rows g * 128). Weights of the first NST steps go out before
      // the wait for the previous kernel (no kernel writes weights); activation
      // tiles after it.
      const int nk = kb1 - kb0;
      const int npre = nk < NST ? nk : NST;
      const uint64_t wpol = l2_evict_first_policy();  // weights: read once per forward
      {
        int tile = kb0 / p.nks, ks = kb0 % p.nks;
        for (int j = 0; j < npre; ++j) {
          mbar_arrive_expect_tx(&full[j], A_BYTES + B_BYTES);
          if (p.w_tiled)
            tma_load_2d_hint(sA + j * A_BYTES, &tmW, &full[j], 0, (kb0 + j) * BM, wpol);
          else
            tma_load_2d_hint(sA + j * A_BYTES, &tmW, &full[j], ks * BK, tile * BM, wpol);
          if (++ks == p.nks) {
            ks = 0;
            ++tile;
          }
        }
      }
      griddep_wait();
      int kc = 0;
      int tile = kb0 / p.nks, ks = kb0 % p.nks;
      for (; kc < nk; ++kc) {
        const int st = kc % NST;
        if (kc >= npre) {
          if (kc >= NST && !mbar_wait(&empty[st], ((kc / NST) - 1) & 1, p.status, abort_flag)) break;
          mbar_arrive_expect_tx(&full[st], A_BYTES + B_BYTES);
          if (p.w_tiled)
            tma_load_2d_hint(sA + st * A_BYTES, &tmW, &full[st], 0, (kb0 + kc) * BM, wpol);
          else
            tma_load_2d_hint(sA + st * A_BYTES, &tmW, &full[st], ks * BK, tile * BM, wpol);
        }
        tma_load_2d(sB + st * B_BYTES, &tmX, &full[st], ks * BK, 0);
        if (++ks == p.nks) {
          ks = 0;
          ++tile;
        }
      }
      if (*abort_flag) {
        for (int j = (kc > NST ? kc - NST : 0); j < kc; ++j) mbar_drain(&full[j % NST], (j / NST) & 1);
        // weights prefetched past the point where the loop stopped
        for (int j = kc; j < npre; ++j) mbar_drain(&full[j], 0);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(BM, MT, false, false);
      const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
      int kc = 0, ic = 0;
      bool ok = true;
      // one accumulator per segment (this CTA's part of one tile)
      for (int g0 = kb0; ok && g0 < kb1; ++ic) {
        const int lo = g0 % p.nks;
        const int hi = (kb1 - g0) < (p.nks - lo) ? lo + (kb1 - g0) : p.nks;
        g0 += hi - lo;
        const int buf = ic & 1;
        if (ic >= 2 && !mbar_wait(&acc_empty[buf], ((ic >> 1) - 1) & 1, p.status, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + buf * MT;
        for (int ks = lo; ks < hi; ++ks) {
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
            umma_f16(d, ad, bd, idesc, (ks > lo || kk > 0) ? 1u : 0u);
          }
          umma_commit(&empty[st]);
          ++kc;
        }
        if (!ok) break;
        umma_commit(&acc_full[buf]);
      }
      // every MMA issued above has finished before TMEM is released
      umma_commit(mma_done);
      mbar_drain(mma_done, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const uint32_t quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int tid = threadIdx.x - 64;
    const uint32_t tl = tmem + ((quarter * 32u) << 16);
    griddep_wait();
    const int G = gridDim.x;
    const int c = blockIdx.x;
    int ic = 0;
    for (int g0 = kb0; g0 < kb1; ++ic) {
      const int tile = g0 / p.nks;
      const int lo = g0 % p.nks;
      const int hi = (kb1 - g0) < (p.nks - lo) ? lo + (kb1 - g0) : p.nks;
      g0 += hi - lo;
      const bool whole = lo == 0 && hi == p.nks;
      // A split tile's contributors are CTAs cf..cl, in k order. Contributor x
      // keeps its partial in slot 0 when its range starts inside the tile (the
      // tile is its first segment), else in slot 1: so cf uses slot 1 (its
      // range holds the tile's first k-step) and every later one slot 0.
      const int t0 = tile * p.nks;
      const int cf = ((t0 + 1) * G - 1) / U;
      const int cl = ((t0 + p.nks) * G - 1) / U;
      const int my_slot = lo > 0 ? 0 : 1;
      const int buf = ic & 1;
      bool ok = mbar_wait(&acc_full[buf], (ic >> 1) & 1, p.status, abort_flag);
      if (!bar_and(ok)) break;
      tc_fence_after();
      if (!ARGMAX && p.mode == GEMM_EPI_PARTIAL) {
        // the partial alone, token-major so that the consumer's reads of a
        // token row are coalesced; no counter, no merge
        float* part = p.ws + (size_t)(c * p.maxseg + ic) * MT * BM + r;
#pragma unroll 1
        for (int sl = 0; sl < MT / 32 && sl * 32 < p.T; ++sl) {
          float v[32];
          tmem_ld32(tl + buf * MT + sl * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (sl * 32 + j < p.T) __stcg(part + (size_t)(sl * 32 + j) * BM, v[j]);
        }
        tc_fence_before();
        mbar_arrive(&acc_empty[buf]);
        continue;
      }
      if constexpr (MT > 64) {
        // 32-column slices (registers): the accumulator stays in TMEM until the
        // segment is done; per column the arithmetic is that of the narrow
        // instances (the same partials, summed in the same order).
        constexpr int NSL = MT / 32;
        bool last = true;
        if (!whole) {
          float4* part = reinterpret_cast<float4*>(p.ws + ((size_t)(c * 2 + my_slot) * BM + r) * MT);
#pragma unroll 1
          for (int sl = 0; sl < NSL && sl * 32 < p.T; ++sl) {
            float v[32];
            tmem_ld32(tl + buf * MT + sl * 32, v);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 8; ++q)
              if (sl * 32 + q * 4 < p.T)
                __stcg(part + sl * 8 + q, make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
          }
          bar_sync128();
          if (tid == 0) {
            int old;
            asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                         : "=r"(old)
                         : "l"(p.counters + tile)
                         : "memory");
            *last_flag = (old == cl - cf) ? 1 : 0;
          }
          bar_sync128();
          last = *last_flag != 0;
        }
        if (last) {
#pragma unroll 1
          for (int sl = 0; sl < NSL && sl * 32 < p.T; ++sl) {
            float v[32];
            tmem_ld32(tl + buf * MT + sl * 32, v);
            tmem_wait_ld();
            if (!whole) {
              float acc[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) acc[j] = 0.f;
              for (int x = cf; x <= cl; ++x) {
                if (x == c) {
#pragma unroll
                  for (int j = 0; j < 32; ++j) acc[j] += v[j];
                  continue;
                }
                const int xs = x == cf ? 1 : 0;
                const float4* src =
                    reinterpret_cast<const float4*>(p.ws + ((size_t)(x * 2 + xs) * BM + r) * MT) + sl * 8;
                float4 t[8];
#pragma unroll
                for (int q = 0; q < 8; ++q)
                  t[q] = (sl * 32 + q * 4 < p.T) ? __ldcg(src + q) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                  acc[4 * q] += t[q].x;
                  acc[4 * q + 1] += t[q].y;
                  acc[4 * q + 2] += t[q].z;
                  acc[4 * q + 3] += t[q].w;
                }
              }
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = acc[j];
            }
            if constexpr (ARGMAX) {
              epilogue_argmax(p, tile, r, lane, quarter, v, sred, MT, sl * 32);
            } else {
              epilogue<32>(p, tile, r, v, sl * 32);
            }
          }
          if (!whole && tid == 0) p.counters[tile] = 0;
        }
        tc_fence_before();
        mbar_arrive(&acc_empty[buf]);
      } else {
        float v[MT];
#pragma unroll
        for (int q = 0; q < MT; q += 32) tmem_ld32(tl + buf * MT + q, v + q);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&acc_empty[buf]);
        if (!whole) {
          // partial layout [CTA][slot][row r][MT token rows]: 16-byte stores
          float4* part = reinterpret_cast<float4*>(p.ws + ((size_t)(c * 2 + my_slot) * BM + r) * MT);
#pragma unroll
          for (int q = 0; q < MT / 4; ++q)
            if (q * 4 < p.T)
              __stcg(part + q, make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
          // The barrier orders the group's partial stores before thread 0's
          // release-acquire increment (cumulative at GPU scope); the last
          // contributor to arrive then sees every other contributor's partial.
          bar_sync128();
          if (tid == 0) {
            int old;
            asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                         : "=r"(old)
                         : "l"(p.counters + tile)
                         : "memory");
            *last_flag = (old == cl - cf) ? 1 : 0;
          }
          bar_sync128();
          if (!*last_flag) continue;
          // sum the contributors in k order (the same additions for every T)
          float acc[MT];
#pragma unroll
          for (int m = 0; m < MT; ++m) acc[m] = 0.f;
          if (p.T <= 4) {
            // one 16-byte partial per contributor: load eight at a time, then add
            for (int x0 = cf; x0 <= cl; x0 += 8) {
              float4 t[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int x = x0 + j;
                t[j] = (x <= cl && x != c)
                           ? __ldcg(reinterpret_cast<const float4*>(
                                 p.ws + ((size_t)(x * 2 + (x == cf ? 1 : 0)) * BM + r) * MT))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
              }
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int x = x0 + j;
                if (x > cl) break;
                const float4 y = x == c ? make_float4(v[0], v[1], v[2], v[3]) : t[j];
                acc[0] += y.x;
                acc[1] += y.y;
                acc[2] += y.z;
                acc[3] += y.w;
              }
            }
          } else {
            for (int x = cf; x <= cl; ++x) {
              if (x == c) {
#pragma unroll
                for (int m = 0; m < MT; ++m) acc[m] += v[m];
                continue;
              }
              const float4* src = reinterpret_cast<const float4*>(
                  p.ws + ((size_t)(x * 2 + (x == cf ? 1 : 0)) * BM + r) * MT);
              float4 t[MT / 4];
#pragma unroll
              for (int q = 0; q < MT / 4; ++q)
                t[q] = (q * 4 < p.T) ? __ldcg(src + q) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
              for (int q = 0; q < MT / 4; ++q) {
                acc[4 * q] += t[q].x;
                acc[4 * q + 1] += t[q].y;
                acc[4 * q + 2] += t[q].z;
                acc[4 * q + 3] += t[q].w;
              }
            }
          }
#pragma unroll
          for (int m = 0; m < MT; ++m) v[m] = acc[m];
          if (tid == 0) p.counters[tile] = 0;
        }
        if constexpr (ARGMAX) {
#pragma unroll
          for (int q = 0; q < MT; q += 32) epilogue_argmax(p, tile, r, lane, quarter, v + q, sred, MT, q);
        } else {
          epilogue<MT>(p, tile, r, v, 0);
        }
      }
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

// Merges the per-tile partials of one token row in tile order: each of the
// 256 threads folds tiles tid, tid + 256, ..., then the threads merge by
// warp shuffles and the warps in order through shared memory.
constexpr int MERGE_THREADS = 256;

__global__ void __launch_bounds__(MERGE_THREADS)
    argmax_merge_kernel(const float4* __restrict__ red, int ntiles, int stride,
                        int32_t* __restrict__ argmax, float* __restrict__ conf) {
  griddep_launch();
  griddep_wait();
  const int t = blockIdx.x;
  Red a{-INFINITY, 0.f, -INFINITY, 0x7fffffff};
  for (int i = threadIdx.x; i < ntiles; i += MERGE_THREADS) {
    const float4 f = __ldcg(red + (size_t)i * stride + t);
    red_merge(a, Red{f.x, f.y, f.z, __float_as_int(f.w)});
  }
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) red_merge(a, red_shfl(a, off));
  __shared__ Red sh[MERGE_THREADS / 32];
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    Red acc = sh[0];
    for (int w = 1; w < MERGE_THREADS / 32; ++w) red_merge(acc, sh[w]);
    if (acc.bi == 0x7fffffff) {
      argmax[t] = -1;
      conf[t] = 0.f;
    } else {
      argmax[t] = acc.bi;
      conf[t] = ex2f((acc.bv - acc.m) * L2E) / acc.s;
    }
  }
}

}  // namespace gemm

ndiff_status launch_argmax_merge(const float4* red, int ntiles, int T, int stride, int32_t* argmax,
                                 float* conf, cudaStream_t stream) {
  if (T <= 0) return NDIFF_OK;
  NDIFF_CUDA_TRY(launch_k(gemm::argmax_merge_kernel, dim3(T), dim3(gemm::MERGE_THREADS), 0, stream,
                          red, ntiles, stride, argmax, conf));
  return NDIFF_OK;
}

GemmPlan gemm_plan(int N, int K) {
  GemmPlan pl;
  pl.ntiles = (N + gemm::BM - 1) / gemm::BM;
  pl.nks = K / gemm::BK;
  // stream-K: one CTA per SM, each an equal contiguous run of the tiles'
  // k-steps (so every SM streams the same number of 16 KB weight tiles)
  const long long U = (long long)pl.ntiles * pl.nks;
  const int sms = num_sms();
  pl.grid = U < sms ? (int)U : sms;
  pl.S = 0;
  pl.nchunks = 1;
  pl.items = pl.ntiles;
  return pl;
}

int gemm_plan_maxseg(const GemmPlan& pl) {
  const long long U = (long long)pl.ntiles * pl.nks;
  const long long run = (U + pl.grid - 1) / pl.grid;  // longest run of k-steps
  return (int)((run + pl.nks - 1) / pl.nks) + 1;
}

size_t gemm_partial_only_bytes(const GemmPlan& pl, int mt) {
  return (size_t)pl.grid * gemm_plan_maxseg(pl) * mt * gemm::BM * sizeof(float);
}

size_t gemm_partials_bytes(const GemmPlan& pl, int mt) {
  // two partial tiles per CTA: its first segment and its last
  return (size_t)pl.grid * 2 * gemm::BM * mt * sizeof(float);
}

ndiff_status gemm_make_maps(const void* w, int N, int K, bool w_tiled, const void* x, int M,
                            CUtensorMap* tmW, CUtensorMap* tmX, int mt) {
  if (tmW) {
    const uint32_t box[2] = {gemm::BK, gemm::BM};
    ndiff_status s;
    if (w_tiled) {
      // [tiles * K/64 * 128][64]: tile (t, ks) is rows (t * K/64 + ks) * 128 ...
      const uint64_t rows = (uint64_t)((N + gemm::BM - 1) / gemm::BM) * (K / gemm::BK) * gemm::BM;
      const uint64_t dims[2] = {(uint64_t)gemm::BK, rows};
      const uint64_t strides[1] = {(uint64_t)gemm::BK * 2};
      s = make_tmap_bf16(tmW, w, 2, dims, strides, box);
    } else {
      const uint64_t dims[2] = {(uint64_t)K, (uint64_t)N};
      const uint64_t strides[1] = {(uint64_t)K * 2};
      s = make_tmap_bf16(tmW, w, 2, dims, strides, box);
    }
    if (s != NDIFF_OK) return s;
  }
  if (tmX) {
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)M};
    const uint64_t strides[1] = {(uint64_t)K * 2};
    const uint32_t box[2] = {gemm::BK, (uint32_t)mt};
    ndiff_status s = make_tmap_bf16(tmX, x, 2, dims, strides, box);
    if (s != NDIFF_OK) return s;
  }
  return NDIFF_OK;
}

template <int MT, bool ARGMAX>
static ndiff_status launch_variant(const CUtensorMap& tmW, const CUtensorMap& tmX, const GemmPlan& pl,
                                   const GemmParams& p, cudaStream_t stream) {
  static bool attr_set[64] = {false};
  int dev = 0;
  NDIFF_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 64 && !attr_set[dev]) {
    NDIFF_CUDA_TRY(cudaFuncSetAttribute(gemm::gemm_bf16_kernel<MT, ARGMAX>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        gemm::Geo<MT>::SMEM_BYTES));
    attr_set[dev] = true;
  }
  NDIFF_CUDA_TRY(launch_k(gemm::gemm_bf16_kernel<MT, ARGMAX>, dim3(pl.grid), dim3(gemm::THREADS),
                          (size_t)gemm::Geo<MT>::SMEM_BYTES, stream, tmW, tmX, p));
  return NDIFF_OK;
}

ndiff_status launch_gemm_bf16(const CUtensorMap& tmW, const CUtensorMap& tmX, const GemmPlan& pl,
                              GemmParams p, cudaStream_t stream, int mt) {
  if (mt != 32 && mt != 64 && mt != 128)
    return set_error(NDIFF_ERR_UNSUPPORTED, "projection kernel: 32, 64 or 128 token rows (got %d)", mt);
  if (p.T > mt) return set_error(NDIFF_ERR_INVALID_ARG, "projection kernel: %d rows > %d", p.T, mt);
  if ((long long)pl.ntiles * pl.nks * (pl.grid + 1) >= (1LL << 31))
    return set_error(NDIFF_ERR_UNSUPPORTED, "projection kernel: %d x %d k-steps is too large",
                     pl.ntiles, pl.nks);
  p.S = 0;
  p.nks = pl.nks;
  p.items = pl.ntiles;
  p.ntiles = pl.ntiles;
  p.status = device_status_word();
  const bool am = p.mode == GEMM_EPI_ARGMAX;
  if (mt == 32)
    return am ? launch_variant<32, true>(tmW, tmX, pl, p, stream)
              : launch_variant<32, false>(tmW, tmX, pl, p, stream);
  if (mt == 64)
    return am ? launch_variant<64, true>(tmW, tmX, pl, p, stream)
              : launch_variant<64, false>(tmW, tmX, pl, p, stream);
  return am ? launch_variant<128, true>(tmW, tmX, pl, p, stream)
            : launch_variant<128, false>(tmW, tmX, pl, p, stream);
}

}  // namespace ndiff
