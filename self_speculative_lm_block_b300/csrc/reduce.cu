// reduce.cu — fused logits reduction: per row, the greedy (temperature-0) id
// and its probability under the full softmax, in one pass over HBM.
//
// Greedy selection is the decision rule under which self-speculation
// reproduces AR output ("NVIDIA 发布 Nemotron-Labs Diffusion 语言模型系列"
// (fintech-frontier-insights), "三种生成模式"); the probability is the confidence
// that orders the diffusion unmask step.
//
// One CTA of 512 threads per row. Each thread streams 16-byte vectors (8 bf16
// or 4 fp32) with four loads in flight, keeping a running maximum m over all
// ids, the sum s of 2^((x - m) log2 e) (rescaled when m grows; one ex2 per
// element) and the best (value, lowest id) over the non-excluded ids. Threads
// merge by warp shuffles, then warps through shared memory.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace ndiff {
namespace {

constexpr int RT = 512;
constexpr float L2E = 1.4426950408889634f;

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct Acc {
  float m;    // running max over all ids
  float s;    // sum of 2^((x - m) * log2 e)
  float bv;   // best value over allowed ids
  int bi;     // its id (INT_MAX: none yet)
};

__device__ __forceinline__ void acc_merge(Acc& a, const Acc& o) {
  const float m = fmaxf(a.m, o.m);
  const float sa = (a.m == -INFINITY) ? 0.f : a.s * ex2f((a.m - m) * L2E);
  const float so = (o.m == -INFINITY) ? 0.f : o.s * ex2f((o.m - m) * L2E);
  a.m = m;
  a.s = sa + so;
  if (o.bv > a.bv || (o.bv == a.bv && o.bi < a.bi)) {
    a.bv = o.bv;
    a.bi = o.bi;
  }
}

template <int N>
__device__ __forceinline__ void acc_vec(Acc& a, const float (&x)[N], int base, int excl) {
  float vmax = x[0];
#pragma unroll
  for (int i = 1; i < N; ++i) vmax = fmaxf(vmax, x[i]);
  if (vmax > a.m) {
    a.s = (a.m == -INFINITY) ? 0.f : a.s * ex2f((a.m - vmax) * L2E);
    a.m = vmax;
  }
  const float nm = -a.m * L2E;
  float t = 0.f;
#pragma unroll
  for (int i = 0; i < N; ++i) t += ex2f(fmaf(x[i], L2E, nm));
  a.s += t;
  if (excl >= base && excl < base + N) {
#pragma unroll
    for (int i = 0; i < N; ++i)
      if (base + i != excl && x[i] > a.bv) {
        a.bv = x[i];
        a.bi = base + i;
      }
  } else if (vmax > a.bv) {
    int idx = N - 1;
#pragma unroll
    for (int i = N - 1; i >= 0; --i)
      if (x[i] == vmax) idx = i;
    a.bv = vmax;
    a.bi = base + idx;
  }
}

__device__ __forceinline__ void unpack8(const uint4& u, float (&x)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <bool BF16>
__global__ void __launch_bounds__(RT) logits_reduce_kernel(const void* __restrict__ logits, int V,
                                                           int64_t ld, int excl,
                                                           int32_t* __restrict__ argmax,
                                                           float* __restrict__ conf) {
  constexpr int EPV = BF16 ? 8 : 4;  // elements per 16-byte vector
  griddep_launch();
  griddep_wait();
  const int r = blockIdx.x;
  const char* row = static_cast<const char*>(logits) + (size_t)r * ld * (BF16 ? 2 : 4);
  const uint4* vrow = reinterpret_cast<const uint4*>(row);
  const int nvec = V / EPV;
  Acc a{-INFINITY, 0.f, -INFINITY, 0x7fffffff};
  int v = threadIdx.x;
  for (; v + 3 * RT < nvec; v += 4 * RT) {
    uint4 u[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) u[k] = __ldcs(vrow + v + k * RT);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float x[EPV];
      if constexpr (BF16) {
        unpack8(u[k], x);
      } else {
        x[0] = __uint_as_float(u[k].x);
        x[1] = __uint_as_float(u[k].y);
        x[2] = __uint_as_float(u[k].z);
        x[3] = __uint_as_float(u[k].w);
      }
      acc_vec<EPV>(a, x, (v + k * RT) * EPV, excl);
    }
  }
  for (; v < nvec; v += RT) {
    const uint4 u = __ldcs(vrow + v);
    float x[EPV];
    if constexpr (BF16) {
      unpack8(u, x);
    } else {
      x[0] = __uint_as_float(u.x);
      x[1] = __uint_as_float(u.y);
      x[2] = __uint_as_float(u.z);
      x[3] = __uint_as_float(u.w);
    }
    acc_vec<EPV>(a, x, v * EPV, excl);
  }
  // ragged tail of fewer than EPV elements
  const int tail0 = nvec * EPV;
  if ((int)threadIdx.x < V - tail0) {
    const int i = tail0 + threadIdx.x;
    float x[1];
    if constexpr (BF16) {
      x[0] = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(row)[i]);
    } else {
      x[0] = reinterpret_cast<const float*>(row)[i];
    }
    acc_vec<1>(a, x, i, excl);
  }
  // warp then block merge
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    Acc o;
    o.m = __shfl_xor_sync(0xffffffffu, a.m, off);
    o.s = __shfl_xor_sync(0xffffffffu, a.s, off);
    o.bv = __shfl_xor_sync(0xffffffffu, a.bv, off);
    o.bi = __shfl_xor_sync(0xffffffffu, a.bi, off);
    acc_merge(a, o);
  }
  __shared__ Acc sh[RT / 32];
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    Acc t = sh[0];
    for (int w = 1; w < RT / 32; ++w) acc_merge(t, sh[w]);
    if (t.bi == 0x7fffffff) {
      argmax[r] = -1;
      conf[r] = 0.f;
    } else {
      argmax[r] = t.bi;
      conf[r] = ex2f((t.bv - t.m) * L2E) / t.s;
    }
  }
}

}  // namespace

ndiff_status launch_logits_reduce(ndiff_dtype dt, const void* logits, int R, int V, int64_t ld,
                                  int exclude_id, int32_t* argmax, float* conf,
                                  cudaStream_t stream) {
  if (R == 0) return NDIFF_OK;
  if (dt == NDIFF_BF16)
    NDIFF_CUDA_TRY(launch_k(logits_reduce_kernel<true>, dim3(R), dim3(RT), 0, stream, logits, V, ld,
                            exclude_id, argmax, conf));
  else
    NDIFF_CUDA_TRY(launch_k(logits_reduce_kernel<false>, dim3(R), dim3(RT), 0, stream, logits, V,
                            ld, exclude_id, argmax, conf));
  return NDIFF_OK;
}

}  // namespace ndiff
