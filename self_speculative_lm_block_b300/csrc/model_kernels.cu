// model_kernels.cu — the small kernels of the random-init tri-mode model:
// weight generation, RoPE table, embedding gather, RMSNorm, the fp32 path's
// projections and epilogues, and the session-state updates of a decode cycle.
//
// Model ("Nemotron-Labs-Diffusion: 一种统一自回归、扩散和自推测解码的三模式语言
// 模型" (ai-feeds.com), "方法": one backbone shared by all modes; "NVIDIA 发布
// Nemotron-Labs Diffusion 语言模型系列" (fintech-frontier-insights), "三种生成
// 模式": one checkpoint, three decode modes). The pages give no weights; the
// model is a pre-norm transformer with every weight drawn N(0, 0.02^2).
//
// Weight stream: element i of tensor t is lane i % 4 of block i / 4 of
// Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
// as 1, 2, 3", SC'11) with counter (i / 4, t, 0, 0) and key (seed, 0); lanes
// 0/1 are the Box-Muller pair (Box & Muller, 1958) of words 0/1, lanes 2/3 the
// pair of words 2/3; the value is float(0.02 * z), then bf16 (nearest even)
// for bf16 models.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"
#include "model_kernels.h"

namespace ndiff {
namespace mk {

// ---------------------------------------------------------------- Philox4x64-10
__device__ __forceinline__ void philox4x64_10(uint64_t& x0, uint64_t& x1, uint64_t& x2,
                                              uint64_t& x3, uint64_t k0, uint64_t k1) {
  const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
  const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
  for (int rnd = 0; rnd < 10; ++rnd) {
    if (rnd) {
      k0 += W0;
      k1 += W1;
    }
    const uint64_t hi0 = __umul64hi(M0, x0), lo0 = M0 * x0;
    const uint64_t hi1 = __umul64hi(M1, x2), lo1 = M1 * x2;
    const uint64_t y0 = hi1 ^ x1 ^ k0, y2 = hi0 ^ x3 ^ k1;
    x0 = y0;
    x1 = lo1;
    x2 = y2;
    x3 = lo0;
  }
}

__device__ __forceinline__ void box_muller(uint64_t wa, uint64_t wb, double& z0, double& z1) {
  const double u1 = ((double)(wa >> 11) + 1.0) * 0x1p-53;
  const double u2 = (double)(wb >> 11) * 0x1p-53;
  const double r = sqrt(-2.0 * log(u1));
  const double th = u2 * 6.283185307179586;
  double s, c;
  sincos(th, &s, &c);
  z0 = r * c;
  z1 = r * s;
}

__device__ __forceinline__ int64_t map_row(int64_t row, int map) {
  if (map == ROWMAP_GATE) return (row / 64) * 128 + 2 * (row % 64);
  if (map == ROWMAP_UP) return (row / 64) * 128 + 2 * (row % 64) + 1;
  if (map == ROWMAP_ROPE) {
    const int64_t i = row % 128;
    return (row / 128) * 128 + (i < 64 ? 2 * i : 2 * (i - 64) + 1);
  }
  return row;
}

// Element (storage row srow, column col) of a weight stored either row-major
// or as contiguous 128 x 64 tiles (tile (srow/128, col/64) at index
// (srow/128) * (cols/64) + col/64, rows of 64 elements inside), the layout
// the projection kernel streams one 16 KB tile at a time.
__device__ __forceinline__ int64_t store_index(int64_t srow, int64_t col, int64_t cols, int tiled) {
  if (!tiled) return srow * cols + col;
  return ((srow / 128) * (cols / 64) + col / 64) * 8192 + (srow % 128) * 64 + (col % 64);
}

__global__ void init_normal_kernel(void* dst, int is_bf16, int tensor_id, int64_t rows,
                                   int64_t cols, int64_t row_off, int map, int tiled, uint64_t seed,
                                   double sigma) {
  const int64_t count = rows * cols;
  const int64_t nblk = (count + 3) / 4;
  for (int64_t n = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; n < nblk;
       n += (int64_t)gridDim.x * blockDim.x) {
    uint64_t w0 = (uint64_t)n, w1 = (uint64_t)tensor_id, w2 = 0, w3 = 0;
    philox4x64_10(w0, w1, w2, w3, seed, 0);
    double z[4];
    box_muller(w0, w1, z[0], z[1]);
    box_muller(w2, w3, z[2], z[3]);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t e = n * 4 + j;
      if (e >= count) break;
      const int64_t row = e / cols, col = e % cols;
      const int64_t at = store_index(map_row(row, map) + row_off, col, cols, tiled);
      const float v = (float)(sigma * z[j]);
      if (is_bf16)
        static_cast<__nv_bfloat16*>(dst)[at] = __float2bfloat16_rn(v);
      else
        static_cast<float*>(dst)[at] = v;
    }
  }
}

__global__ void gather_weight_kernel(const void* src, int is_bf16, int64_t cols, int64_t row_off,
                                     int map, int tiled, int64_t offset, int64_t count, float* out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = offset + i;
    const int64_t row = e / cols, col = e % cols;
    const int64_t at = store_index(map_row(row, map) + row_off, col, cols, tiled);
    out[i] = is_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(src)[at])
                     : static_cast<const float*>(src)[at];
  }
}

// (cos, sin) of pos * base^(-2i/D) for pos < Lmax, i < D/2; double precision.
__global__ void rope_table_kernel(float2* tab, int Lmax, int D, double base) {
  const int half = D / 2;
  const int64_t total = (int64_t)Lmax * half;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int pos = (int)(e / half), i = (int)(e % half);
    const double inv = pow(base, -(2.0 * i) / D);
    double s, c;
    sincos((double)pos * inv, &s, &c);
    tab[e] = make_float2((float)c, (float)s);
  }
}

// ---------------------------------------------------------------- activations
template <bool BF16>
__global__ void embed_kernel(const void* E, const int32_t* ids, int V, int d, float* x,
                             unsigned int* status) {
  griddep_launch();
  griddep_wait();
  const int m = blockIdx.x;
  int id = ids[m];
  if (id < 0 || id >= V) {  // reported, and clamped only to keep the read in bounds
    if (threadIdx.x == 0 && status != nullptr) atomicOr(status, kStatusBadInput);
    id = id < 0 ? 0 : V - 1;
  }
  for (int k = threadIdx.x; k < d; k += blockDim.x) {
    const size_t at = (size_t)id * d + k;
    x[(size_t)m * d + k] = BF16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(E)[at])
                                : static_cast<const float*>(E)[at];
  }
}

// h = x / sqrt(mean(x^2) + eps), one CTA of 256 threads per row, fixed
// summation order (a row's result does not depend on the other rows).
template <bool BF16>
__global__ void __launch_bounds__(256) rmsnorm_kernel(const float* x, int d, float eps, void* out) {
  griddep_launch();
  griddep_wait();
  const int m = blockIdx.x;
  const float* xr = x + (size_t)m * d;
  float ss = 0.f;
  for (int k = threadIdx.x; k < d; k += 256) ss = fmaf(xr[k], xr[k], ss);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  __shared__ float part[8];
  __shared__ float inv_s;
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < 8; ++w) t += part[w];
    inv_s = 1.f / sqrtf(t / (float)d + eps);
  }
  __syncthreads();
  const float inv = inv_s;
  for (int k = threadIdx.x; k < d; k += 256) {
    const float v = xr[k] * inv;
    if (BF16)
      static_cast<__nv_bfloat16*>(out)[(size_t)m * d + k] = __float2bfloat16_rn(v);
    else
      static_cast<float*>(out)[(size_t)m * d + k] = v;
  }
}

// ---------------------------------------------------------------- partial tiles
// Consumers of a projection that left its partial tiles unsummed
// (GEMM_EPI_PARTIAL). Tile t of a stream-K partition (U k-steps over G CTAs,
// nks k-steps a tile) is covered by CTAs cf..cl in k order; CTA c keeps its
// segment of tile t in slot c * maxseg + (t - start(c) / nks), start(c) =
// c * U / G. A tile's partials are summed in contributor order, the first
// RR_BATCH of them loaded together (16 bytes a lane: 4 tile rows of one token
// row). These sums are the same for every token row and every row count.
constexpr int RR_BATCH = 6;

template <int MT>
__device__ __forceinline__ float4 tile_sum4(const PartialPlan& pp, int t, int m, int row4) {
  const int t0 = t * pp.nks;
  const int cf = ((t0 + 1) * pp.G - 1) / pp.U, cl = ((t0 + pp.nks) * pp.G - 1) / pp.U;
  auto at = [&](int c) {
    const int s = t - (c * pp.U / pp.G) / pp.nks;
    return reinterpret_cast<const float4*>(pp.part + ((size_t)(c * pp.maxseg + s) * MT + m) * 128 + row4);
  };
  float4 pv[RR_BATCH];
#pragma unroll
  for (int j = 0; j < RR_BATCH; ++j) pv[j] = cf + j <= cl ? __ldcg(at(cf + j)) : make_float4(0.f, 0.f, 0.f, 0.f);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 0; j < RR_BATCH; ++j) {
    if (cf + j <= cl) {
      acc.x += pv[j].x;
      acc.y += pv[j].y;
      acc.z += pv[j].z;
      acc.w += pv[j].w;
    }
  }
  for (int c = cf + RR_BATCH; c <= cl; ++c) {  // tiles with more contributors
    const float4 q = __ldcg(at(c));
    acc.x += q.x;
    acc.y += q.y;
    acc.z += q.z;
    acc.w += q.w;
  }
  return acc;
}

// Residual add of the output / down projection fused with the RMSNorm that
// follows: for token row m,
//   x[m][n] += the summed partial of column n,  h[m] = bf16(x[m] / rms(x[m])).
// One CTA per row, one warp per 128-column tile (up to 32 warps; warp w also
// takes tiles w + 32, ...), lane l on columns 4l .. 4l+3. The sum of squares
// runs lane, warp-shuffle tree, warps in order. Requires d % 128 == 0.
template <int MT>
__global__ void __launch_bounds__(1024)
    residual_rmsnorm_kernel(float* __restrict__ x, int d, float eps, __nv_bfloat16* __restrict__ h,
                            const PartialPlan pp) {
  griddep_launch();
  griddep_wait();
  const int m = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int ntile = d >> 7;
  float* xr = x + (size_t)m * d;
  float ss = 0.f;
  float4 keep0 = make_float4(0.f, 0.f, 0.f, 0.f), keep1 = keep0;  // a warp's first two tiles
  int it = 0;
  for (int t = warp; t < ntile; t += nw, ++it) {  // uniform over the warp
    float4* xp = reinterpret_cast<float4*>(xr + t * 128 + lane * 4);
    const float4 xo = *xp;
    const float4 acc = tile_sum4<MT>(pp, t, m, lane * 4);
    const float4 v = make_float4(xo.x + acc.x, xo.y + acc.y, xo.z + acc.z, xo.w + acc.w);
    *xp = v;
    if (it == 0) keep0 = v;
    if (it == 1) keep1 = v;
    ss = fmaf(v.x, v.x, ss);
    ss = fmaf(v.y, v.y, ss);
    ss = fmaf(v.z, v.z, ss);
    ss = fmaf(v.w, v.w, ss);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  __shared__ float wsum[32];
  __shared__ float inv_s;
  if (lane == 0) wsum[warp] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < nw; ++w) t += wsum[w];
    inv_s = 1.f / sqrtf(t / (float)d + eps);
  }
  __syncthreads();
  const float inv = inv_s;
  it = 0;
  for (int t = warp; t < ntile; t += nw, ++it) {
    const float4 v = it == 0 ? keep0 : (it == 1 ? keep1 : *reinterpret_cast<const float4*>(xr + t * 128 + lane * 4));
    uint2 o;
    o.x = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.x * inv)) |
          ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.y * inv)) << 16);
    o.y = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.z * inv)) |
          ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.w * inv)) << 16);
    *reinterpret_cast<uint2*>(h + (size_t)m * d + t * 128 + lane * 4) = o;
  }
}

// residual_rmsnorm_kernel for a few token rows (an AR step) with the row
// spread over a cluster of C CTAs (blockIdx.x = rank), one warp a tile, so
// that the row's ~100 KB of loads (x and the partials at d = 4096) are taken
// by C SMs instead of one. For d / 128 <= 32 tiles, where the one-CTA kernel
// gives each warp one tile, the arithmetic is that kernel's: the tiles' sums
// of squares are added in tile order (warp 0 of every CTA reads all of them
// from the cluster's shared memory after a cluster barrier), so a row's
// result does not depend on which kernel ran it.
template <int MT>
__global__ void __launch_bounds__(256)
    residual_rmsnorm_cluster_kernel(float* __restrict__ x, int d, float eps, __nv_bfloat16* __restrict__ h,
                                    const PartialPlan pp) {
  griddep_launch();
  griddep_wait();
  const int m = blockIdx.y, rank = blockIdx.x;  // the cluster spans the grid's x
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int ntile = d >> 7;
  const int t = rank * nw + warp;
  float4* xp = reinterpret_cast<float4*>(x + (size_t)m * d + t * 128 + lane * 4);
  const float4 xo = *xp;
  const float4 acc = tile_sum4<MT>(pp, t, m, lane * 4);
  const float4 v = make_float4(xo.x + acc.x, xo.y + acc.y, xo.z + acc.z, xo.w + acc.w);
  *xp = v;
  float ss = 0.f;
  ss = fmaf(v.x, v.x, ss);
  ss = fmaf(v.y, v.y, ss);
  ss = fmaf(v.z, v.z, ss);
  ss = fmaf(v.w, v.w, ss);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  __shared__ float wsum[8];
  __shared__ float inv_s;
  if (lane == 0) wsum[warp] = ss;
  cluster_sync_all();  // every tile's sum is in its CTA's shared memory
  if (warp == 0) {
    const float tv = lane < ntile ? ld_cluster_f32(smem_u32(&wsum[lane % nw]), lane / nw) : 0.f;
    float tv_all[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) tv_all[j] = __shfl_sync(0xffffffffu, tv, j);
    float tot = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < ntile) tot += tv_all[j];
    if (lane == 0) inv_s = 1.f / sqrtf(tot / (float)d + eps);
  }
  __syncthreads();
  const float inv = inv_s;
  uint2 o;
  o.x = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.x * inv)) |
        ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.y * inv)) << 16);
  o.y = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.z * inv)) |
        ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.w * inv)) << 16);
  *reinterpret_cast<uint2*>(h + (size_t)m * d + t * 128 + lane * 4) = o;
  cluster_sync_all();  // no CTA leaves while another still reads its sums
}

// SwiGLU of the gate/up projection: tile rows 2i and 2i+1 hold gate j and up j
// (j = tile * 64 + i); act[m][j] = bf16(silu(g) * u), the expression of the
// projection kernel's SwiGLU epilogue. Grid (tiles / 8, token rows), one warp
// a tile, lane l on rows 4l .. 4l+3 (two gate/up pairs).
template <int MT>
__global__ void __launch_bounds__(256)
    swiglu_merge_kernel(const PartialPlan pp, int ntile, __nv_bfloat16* __restrict__ act, int64_t lda) {
  griddep_launch();
  griddep_wait();
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5), m = blockIdx.y, lane = threadIdx.x & 31;
  if (t >= ntile) return;
  const float4 y = tile_sum4<MT>(pp, t, m, lane * 4);
  const float a0 = y.x / (1.f + expf(-y.x)) * y.y;
  const float a1 = y.z / (1.f + expf(-y.z)) * y.w;
  const uint32_t o = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a0)) |
                     ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a1)) << 16);
  *reinterpret_cast<uint32_t*>(act + (size_t)m * lda + t * 64 + lane * 2) = o;
}

// QKV of one sequence: tile h is one head (q heads, then k, then v). In q and
// k heads rows 2i / 2i+1 hold dims i / i+64 (the RoPE pair) and are rotated
// by the position's (cos, sin) with the expressions of the projection
// kernel's QKV epilogue; v rows are dims in order. q goes to q[m][h][128], k
// and v to the caches at the token's cache row. Positions and cache rows:
// kv_len[0] + m, or with blk_pos those of the token's 32-row block. Grid
// (heads, token rows / R), R = min(T, 8) warps a CTA, one per token row; lane
// l on rows 4l .. 4l+3.
template <int MT>
__global__ void __launch_bounds__(256)
    qkv_merge_kernel(const PartialPlan pp, int T, int Hq, int Hkv, int Lmax, const int32_t* kv_len,
                     const int32_t* blk_pos, const float2* __restrict__ rope,
                     __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ kc,
                     __nv_bfloat16* __restrict__ vc, unsigned int* status) {
  // Dependents launch only once the QKV projection (and so, through the
  // chain of waits, every kernel before it) has completed: the attention
  // after this kernel then reads kv_len and streams the prefix K/V before
  // its own wait.
  griddep_wait();
  griddep_launch();
  const int h = blockIdx.x, lane = threadIdx.x & 31;
  const int m = blockIdx.y * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (m >= T) return;  // uniform over the warp
  // the partials' loads go out first: they do not wait for the position
  const float4 y = tile_sum4<MT>(pp, h, m, lane * 4);
  const int P = checked_prefix(kv_len[0], Lmax - T, status);
  const int pos = blk_pos != nullptr ? blk_pos[2 * (m >> 5)] + (m & 31) : P + m;
  const int slot = blk_pos != nullptr ? blk_pos[2 * (m >> 5) + 1] + (m & 31) : P + m;
  if (h < Hq + Hkv) {
    // rows 4l, 4l+1: dims 2l, 2l+64; rows 4l+2, 4l+3: dims 2l+1, 2l+65
    const float4 cs = __ldg(reinterpret_cast<const float4*>(rope + (size_t)pos * 64 + 2 * lane));
    const float e0 = y.x * cs.x - y.y * cs.y, o0 = y.y * cs.x + y.x * cs.y;
    const float e1 = y.z * cs.z - y.w * cs.w, o1 = y.w * cs.z + y.z * cs.w;
    __nv_bfloat16* dst = h < Hq ? q + ((size_t)m * Hq + h) * 128
                                : kc + ((size_t)(h - Hq) * Lmax + slot) * 128;
    const uint32_t lo = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(e0)) |
                        ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(e1)) << 16);
    const uint32_t hi = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(o0)) |
                        ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(o1)) << 16);
    *reinterpret_cast<uint32_t*>(dst + 2 * lane) = lo;
    *reinterpret_cast<uint32_t*>(dst + 64 + 2 * lane) = hi;
  } else {
    __nv_bfloat16* dst = vc + ((size_t)(h - Hq - Hkv) * Lmax + slot) * 128 + 4 * lane;
    uint2 o;
    o.x = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(y.x)) |
          ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(y.y)) << 16);
    o.y = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(y.z)) |
          ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(y.w)) << 16);
    *reinterpret_cast<uint2*>(dst) = o;
  }
}

// y[m][n] = sum_k x[m][k] W[n][k] in fp32: one warp per (n, m), lane-strided
// partial sums merged by a fixed shuffle tree.
__global__ void __launch_bounds__(256) linear_f32_kernel(const float* x, int ldx, const float* W,
                                                         int N, int K, float* y, int ldy) {
  griddep_launch();
  griddep_wait();
  const int n = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int m = blockIdx.y;
  const int lane = threadIdx.x & 31;
  if (n >= N) return;
  const float* xr = x + (size_t)m * ldx;
  const float* wr = W + (size_t)n * K;
  float acc = 0.f;
  for (int k = lane; k < K; k += 32) acc = fmaf(xr[k], wr[k], acc);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) y[(size_t)m * ldy + n] = acc;
}

// fp32 QKV epilogue: rotate-half RoPE on q and k heads, q to qb [T][Hq][D],
// k and v to the caches [Hkv][Lmax][D] at positions P + m.
__global__ void qkv_rope_f32_kernel(const float* y, int T, int Hq, int Hkv, int D, int Lmax,
                                    const int32_t* kv_len, const float2* rope, float* qb,
                                    float* kc, float* vc, unsigned int* status) {
  griddep_launch();
  griddep_wait();
  const int Ntot = (Hq + 2 * Hkv) * D;
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= T * Ntot) return;
  const int m = e / Ntot, c = e % Ntot, h = c / D, d = c % D, half = D / 2;
  const int P = checked_prefix(kv_len[0], Lmax - T, status);
  const float* yr = y + (size_t)m * Ntot + (size_t)h * D;
  float v = yr[d];
  if (h < Hq + Hkv) {
    const float2 cs = rope[(size_t)(P + m) * half + (d % half)];
    v = d < half ? v * cs.x - yr[d + half] * cs.y : v * cs.x + yr[d - half] * cs.y;
  }
  if (h < Hq)
    qb[((size_t)m * Hq + h) * D + d] = v;
  else if (h < Hq + Hkv)
    kc[((size_t)(h - Hq) * Lmax + P + m) * D + d] = v;
  else
    vc[((size_t)(h - Hq - Hkv) * Lmax + P + m) * D + d] = v;
}

__global__ void swiglu_f32_kernel(const float* y, int T, int ffn, float* a) {
  griddep_launch();
  griddep_wait();
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= T * ffn) return;
  const int m = e / ffn, j = e % ffn;
  const float g = y[(size_t)m * 2 * ffn + j], u = y[(size_t)m * 2 * ffn + ffn + j];
  a[e] = g / (1.f + expf(-g)) * u;
}

__global__ void resid_add_f32_kernel(float* x, const float* y, int n) {
  griddep_launch();
  griddep_wait();
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e < n) x[e] += y[e];
}

// ---------------------------------------------------------------- decode state
// A fresh draft block: slot 0 holds the pending token, slots 1..T-1 [MASK];
// every slot masked, no draft yet.
// Start of a drafted block, one CTA per sequence b: input [last_b, MASK ...],
// no slot fixed yet, every slot masked.
__global__ void block_init_kernel(int32_t* block_in, int32_t* draft, uint32_t* mask, int T,
                                  const int32_t* last, int32_t mask_id) {
  griddep_launch();
  griddep_wait();
  const int b = blockIdx.x, i = threadIdx.x;
  if (i < T) {
    block_in[(size_t)b * T + i] = i == 0 ? last[b] : mask_id;
    draft[(size_t)b * T + i] = -1;
  }
  if (i == 0) mask[b] = T >= 32 ? 0xffffffffu : ((1u << T) - 1u);
}

// End of a decode cycle, one thread per sequence b: the pending token becomes
// the last committed one (tokens[b * stride + n - 1], n = n_ptr[b] or n_const)
// and the committed prefix grows by kv_add (0 when verification has already
// advanced it).
__global__ void commit_kernel(const int32_t* tokens, int stride, const int32_t* n_ptr, int n_const,
                              int kv_add, int32_t* last, int32_t* kv_len, int B) {
  griddep_launch();
  griddep_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int n = n_ptr ? n_ptr[b] : n_const;
  last[b] = tokens[(size_t)b * stride + (n > 0 ? n - 1 : 0)];
  kv_len[b] += kv_add;
}

__global__ void set_token_kernel(int32_t* ids, int32_t tok) {
  griddep_launch();
  griddep_wait();
  ids[0] = tok;
}

__global__ void kv_add_kernel(int32_t* kv_len, int add) {
  griddep_launch();
  griddep_wait();
  kv_len[0] += add;
}

// Fused verify + draft forward of one sequence. fused_input: the 64 input
// tokens [last, d0..d30] (the block under verification, from block_in) and
// [d31, MASK x 31] (the next block to draft), and the draft half's prefix
// kv_len + 32. fused_stash: when the whole block was accepted, the draft
// half's argmaxes become the next block's draft and its verification input
// [d31, d'0..d'30].
__global__ void fused_input_kernel(int32_t* fin, const int32_t* block_in, const int32_t* draft,
                                   int32_t mask_id, const int32_t* kv_len, int32_t* kv_len2) {
  griddep_launch();
  griddep_wait();
  const int i = threadIdx.x;
  if (i < 32) fin[i] = block_in[i];
  else if (i < 64) fin[i] = i == 32 ? draft[31] : mask_id;
  if (i == 0) kv_len2[0] = kv_len[0] + 32;
}

__global__ void fused_stash_kernel(const int32_t* pred2, const int32_t* acclen, const int32_t* last,
                                   int32_t* draft, int32_t* block_in) {
  griddep_launch();
  griddep_wait();
  const int i = threadIdx.x;
  if (acclen[0] != 32 || i >= 32) return;
  draft[i] = pred2[i];
  if (i == 0) block_in[0] = last[0];
  if (i <= 30) block_in[i + 1] = pred2[i];
}

// Quadratic forward of one sequence (128 rows): the block under verification
// [last, d0..d30] at prefix P, the next block [d31, MASK x 31] for full
// acceptance at prefix P + 32, and for each candidate acceptance length c
// (cand[0], cand[1]) a block of 32 [MASK] at prefix P_c = P + c + 1. The
// candidate blocks' K/V go to cache rows past both blocks: S_c = align64(P +
// 64) + 128 (c index), and the attention finds their keys there (remap
// {x_c = P_c rounded down to 64, S_c}); blk_pos gives the QKV epilogue each
// block's first position and cache row.
__global__ void quad_input_kernel(int32_t* fin, const int32_t* block_in, const int32_t* draft,
                                  int32_t mask_id, const int32_t* kv_len, const int32_t* cand,
                                  int32_t* kvc, int4* remap, int32_t* blk_pos) {
  griddep_launch();
  griddep_wait();
  const int i = threadIdx.x;
  if (i < 32) fin[i] = block_in[i];
  else if (i < 128) fin[i] = i == 32 ? draft[31] : mask_id;
  if (i == 0) {
    const int P = kv_len[0];
    const int S0 = (P + 64 + 63) & ~63;
    kvc[0] = P + 32;
    remap[0] = make_int4(kNoRemap, 0, 0, 0);
    blk_pos[0] = P;
    blk_pos[1] = P;
    blk_pos[2] = P + 32;
    blk_pos[3] = P + 32;
    for (int c = 0; c < 2; ++c) {
      const int Pc = P + cand[c] + 1;
      const int x = Pc & ~63, S = S0 + 128 * c;
      kvc[1 + c] = Pc;
      remap[1 + c] = make_int4(x, S, 0, 0);
      blk_pos[4 + 2 * c] = Pc;
      blk_pos[5 + 2 * c] = S + (Pc - x);
    }
  }
}

// After verification: the draft block of the verified acceptance length (32,
// cand[0], cand[1], in that order), if any, becomes the next draft and its
// verification input [last, d'0..d'30].
__global__ void quad_stash_kernel(const int32_t* pred, const int32_t* acclen, const int32_t* cand,
                                  const int32_t* last, int32_t* draft, int32_t* block_in) {
  griddep_launch();
  griddep_wait();
  const int i = threadIdx.x;
  const int L = acclen[0];
  const int src = L == 32 ? 32 : (L == cand[0] ? 64 : (L == cand[1] ? 96 : -1));
  if (src < 0 || i >= 32) return;
  draft[i] = pred[src + i];
  if (i == 0) block_in[0] = last[0];
  if (i <= 30) block_in[i + 1] = pred[src + i];
}

}  // namespace mk

// ---------------------------------------------------------------- launchers
static int grid_for(int64_t work, int threads) {
  const int64_t cap = (int64_t)num_sms() * 16;
  int64_t g = (work + threads - 1) / threads;
  if (g > cap) g = cap;
  return (int)(g < 1 ? 1 : g);
}

ndiff_status launch_init_normal(void* dst, bool bf16, int tensor_id, int64_t rows, int64_t cols,
                                int64_t row_off, int map, bool tiled, uint64_t seed, double sigma,
                                cudaStream_t s) {
  const int64_t nblk = (rows * cols + 3) / 4;
  mk::init_normal_kernel<<<grid_for(nblk, 256), 256, 0, s>>>(dst, bf16 ? 1 : 0, tensor_id, rows,
                                                             cols, row_off, map, tiled ? 1 : 0,
                                                             seed, sigma);
  NDIFF_CUDA_TRY(cudaGetLastError());
  return NDIFF_OK;
}

ndiff_status launch_gather_weight(const void* src, bool bf16, int64_t cols, int64_t row_off,
                                  int map, bool tiled, int64_t offset, int64_t count, float* out,
                                  cudaStream_t s) {
  if (count <= 0) return NDIFF_OK;
  mk::gather_weight_kernel<<<grid_for(count, 256), 256, 0, s>>>(src, bf16 ? 1 : 0, cols, row_off,
                                                                map, tiled ? 1 : 0, offset, count,
                                                                out);
  NDIFF_CUDA_TRY(cudaGetLastError());
  return NDIFF_OK;
}

ndiff_status launch_rope_table(float2* tab, int Lmax, int D, double base, cudaStream_t s) {
  mk::rope_table_kernel<<<grid_for((int64_t)Lmax * (D / 2), 256), 256, 0, s>>>(tab, Lmax, D, base);
  NDIFF_CUDA_TRY(cudaGetLastError());
  return NDIFF_OK;
}

ndiff_status launch_embed(const void* E, bool bf16, const int32_t* ids, int T, int V, int d,
                          float* x, cudaStream_t s) {
  if (bf16)
    NDIFF_CUDA_TRY(launch_k(mk::embed_kernel<true>, dim3(T), dim3(256), 0, s, E, ids, V, d, x,
                            device_status_word()));
  else
    NDIFF_CUDA_TRY(launch_k(mk::embed_kernel<false>, dim3(T), dim3(256), 0, s, E, ids, V, d, x,
                            device_status_word()));
  return NDIFF_OK;
}

#define NDIFF_MT_DISPATCH(KERNEL, MT, GRID, BLOCK, ...)                                     \
  do {                                                                                     \
    if ((MT) == 32)                                                                        \
      NDIFF_CUDA_TRY(launch_k(KERNEL<32>, GRID, BLOCK, 0, s, __VA_ARGS__));               \
    else if ((MT) == 64)                                                                   \
      NDIFF_CUDA_TRY(launch_k(KERNEL<64>, GRID, BLOCK, 0, s, __VA_ARGS__));               \
    else if ((MT) == 128)                                                                  \
      NDIFF_CUDA_TRY(launch_k(KERNEL<128>, GRID, BLOCK, 0, s, __VA_ARGS__));              \
    else                                                                                   \
      return set_error(NDIFF_ERR_UNSUPPORTED, "partial tiles of %d token columns", (MT)); \
  } while (0)

ndiff_status launch_residual_rmsnorm(float* x, int T, int d, float eps, __nv_bfloat16* h,
                                     const PartialPlan& pp, int mt, cudaStream_t s) {
  if (T <= 0) return NDIFF_OK;
  if (d % 128 != 0)
    return set_error(NDIFF_ERR_UNSUPPORTED, "residual_rmsnorm: d_model %d is not a multiple of 128", d);
  const int ntile = d / 128;
  if (mt == 32 && T <= 4 && ntile <= 32 && ntile % 8 == 0) {
    // an AR step: the row over a cluster of 8 CTAs, ntile / 8 warps each
    NDIFF_CUDA_TRY(launch_k_cluster(mk::residual_rmsnorm_cluster_kernel<32>, dim3(8, T), dim3(32 * (ntile / 8)),
                                    0, s, 8, x, d, eps, h, pp));
    return NDIFF_OK;
  }
  const int threads = ntile * 32 < 1024 ? ntile * 32 : 1024;
  NDIFF_MT_DISPATCH(mk::residual_rmsnorm_kernel, mt, dim3(T), dim3(threads), x, d, eps, h, pp);
  return NDIFF_OK;
}

ndiff_status launch_swiglu_merge(const PartialPlan& pp, int ntile, int T, __nv_bfloat16* act, int64_t lda,
                                 int mt, cudaStream_t s) {
  if (T <= 0) return NDIFF_OK;
  NDIFF_MT_DISPATCH(mk::swiglu_merge_kernel, mt, dim3((ntile + 7) / 8, T), dim3(256), pp, ntile, act, lda);
  return NDIFF_OK;
}

ndiff_status launch_qkv_merge(const PartialPlan& pp, int T, int Hq, int Hkv, int Lmax,
                              const int32_t* kv_len, const int32_t* blk_pos, const float2* rope,
                              __nv_bfloat16* q, __nv_bfloat16* kc, __nv_bfloat16* vc, int mt,
                              cudaStream_t s) {
  if (T <= 0) return NDIFF_OK;
  // one warp per (head, token row), up to 8 rows a CTA: a 32-row block is 192
  // CTAs of 8 warps rather than 1536 of one
  const int rows = T < 8 ? T : 8;
  NDIFF_MT_DISPATCH(mk::qkv_merge_kernel, mt, dim3(Hq + 2 * Hkv, (T + rows - 1) / rows), dim3(32 * rows), pp, T,
                    Hq, Hkv, Lmax,
                    kv_len, blk_pos, rope, q, kc, vc, device_status_word());
  return NDIFF_OK;
}

ndiff_status launch_rmsnorm(const float* x, int T, int d, float eps, void* out, bool bf16,
                            cudaStream_t s) {
  if (bf16)
    NDIFF_CUDA_TRY(launch_k(mk::rmsnorm_kernel<true>, dim3(T), dim3(256), 0, s, x, d, eps, out));
  else
    NDIFF_CUDA_TRY(launch_k(mk::rmsnorm_kernel<false>, dim3(T), dim3(256), 0, s, x, d, eps, out));
  return NDIFF_OK;
}

ndiff_status launch_linear_f32(const float* x, int ldx, const float* W, int N, int K, float* y,
                               int ldy, int T, cudaStream_t s) {
  dim3 grid((N + 7) / 8, T);
  mk::linear_f32_kernel<<<grid, 256, 0, s>>>(x, ldx, W, N, K, y, ldy);
  NDIFF_CUDA_TRY(cudaGetLastError());
  return NDIFF_OK;
}

ndiff_status launch_qkv_rope_f32(const float* y, int T, int Hq, int Hkv, int D, int Lmax,
                                 const int32_t* kv_len, const float2* rope, float* qb, float* kc,
                                 float* vc, cudaStream_t s) {
  const int n = T * (Hq + 2 * Hkv) * D;
  mk::qkv_rope_f32_kernel<<<(n + 255) / 256, 256, 0, s>>>(y, T, Hq, Hkv, D, Lmax, kv_len, rope,
                                                          qb, kc, vc, device_status_word());
  NDIFF_CUDA_TRY(cudaGetLastError());
  return NDIFF_OK;
}

ndiff_status launch_swiglu_f32(const float* y, int T, int ffn, float* a, cudaStream_t s) {
  const int n = T * ffn;
  mk::swiglu_f32_kernel<<<(n + 255) / 256, 256, 0, s>>>(y, T, ffn, a);
  NDIFF_CUDA_TRY(cudaGetLastError());
  return NDIFF_OK;
}

ndiff_status launch_resid_add_f32(float* x, const float* y, int n, cudaStream_t s) {
  mk::resid_add_f32_kernel<<<(n + 255) / 256, 256, 0, s>>>(x, y, n);
  NDIFF_CUDA_TRY(cudaGetLastError());
  return NDIFF_OK;
}

ndiff_status launch_commit(const int32_t* tokens, int stride, const int32_t* n_ptr, int n_const,
                           int kv_add, int32_t* last, int32_t* kv_len, int B, cudaStream_t s) {
  NDIFF_CUDA_TRY(launch_k(mk::commit_kernel, dim3((B + 127) / 128), dim3(128), 0, s, tokens, stride,
                          n_ptr, n_const, kv_add, last, kv_len, B));
  return NDIFF_OK;
}

ndiff_status launch_block_init(int32_t* block_in, int32_t* draft, uint32_t* mask, int T,
                               const int32_t* last, int32_t mask_id, int B, cudaStream_t s) {
  NDIFF_CUDA_TRY(launch_k(mk::block_init_kernel, dim3(B), dim3(32), 0, s, block_in, draft, mask, T,
                          last, mask_id));
  return NDIFF_OK;
}

ndiff_status launch_set_token(int32_t* ids, int32_t tok, cudaStream_t s) {
  NDIFF_CUDA_TRY(launch_k(mk::set_token_kernel, dim3(1), dim3(1), 0, s, ids, tok));
  return NDIFF_OK;
}

ndiff_status launch_kv_add(int32_t* kv_len, int add, cudaStream_t s) {
  NDIFF_CUDA_TRY(launch_k(mk::kv_add_kernel, dim3(1), dim3(1), 0, s, kv_len, add));
  return NDIFF_OK;
}

ndiff_status launch_fused_input(int32_t* fin, const int32_t* block_in, const int32_t* draft,
                                int32_t mask_id, const int32_t* kv_len, int32_t* kv_len2,
                                cudaStream_t s) {
  NDIFF_CUDA_TRY(launch_k(mk::fused_input_kernel, dim3(1), dim3(64), 0, s, fin, block_in, draft,
                          mask_id, kv_len, kv_len2));
  return NDIFF_OK;
}

ndiff_status launch_quad_input(int32_t* fin, const int32_t* block_in, const int32_t* draft,
                               int32_t mask_id, const int32_t* kv_len, const int32_t* cand,
                               int32_t* kvc, int4* remap, int32_t* blk_pos, cudaStream_t s) {
  NDIFF_CUDA_TRY(launch_k(mk::quad_input_kernel, dim3(1), dim3(128), 0, s, fin, block_in, draft,
                          mask_id, kv_len, cand, kvc, remap, blk_pos));
  return NDIFF_OK;
}

ndiff_status launch_quad_stash(const int32_t* pred, const int32_t* acclen, const int32_t* cand,
                               const int32_t* last, int32_t* draft, int32_t* block_in,
                               cudaStream_t s) {
  NDIFF_CUDA_TRY(launch_k(mk::quad_stash_kernel, dim3(1), dim3(32), 0, s, pred, acclen, cand, last,
                          draft, block_in));
  return NDIFF_OK;
}

ndiff_status launch_fused_stash(const int32_t* pred2, const int32_t* acclen, const int32_t* last,
                                int32_t* draft, int32_t* block_in, cudaStream_t s) {
  NDIFF_CUDA_TRY(launch_k(mk::fused_stash_kernel, dim3(1), dim3(32), 0, s, pred2, acclen, last,
                          draft, block_in));
  return NDIFF_OK;
}

}  // namespace ndiff
