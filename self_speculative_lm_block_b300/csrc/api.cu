// api.cu — the C ABI of libndiff: status reporting, argument validation and
// dispatch of the decode-step primitives (block attention, logits reduction,
// unmask, verify/accept). The model entry points live in model.cu.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {
thread_local char g_last_error[512] = "";
thread_local bool g_pdl = false;
__device__ unsigned int g_status_word;

struct DeviceCache {
  void* ctx = nullptr;            // the context the addresses below belong to
  unsigned int* status = nullptr;
  int sms = 0;
};
DeviceCache g_dev[64];
std::mutex g_dev_mu;
}  // namespace

namespace ndiff {

bool pdl_enabled() { return g_pdl; }
PdlScope::PdlScope(bool on) : prev(g_pdl) { g_pdl = on; }
PdlScope::~PdlScope() { g_pdl = prev; }

ndiff_status set_error(ndiff_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

ndiff_status cuda_error(cudaError_t e, const char* what) {
  return set_error(NDIFF_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

void* current_context() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  CUcontext c = nullptr;
  if (fn == nullptr || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

// The status word's address and the SM count of the current device, looked
// up again whenever the current context is not the one they were taken in.
static DeviceCache* dev_cache() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceCache& c = g_dev[dev];
  void* ctx = current_context();
  if (c.status == nullptr || ctx == nullptr || ctx != c.ctx) {
    void* p = nullptr;
    c.status = cudaGetSymbolAddress(&p, g_status_word) == cudaSuccess ? (unsigned int*)p : nullptr;
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    c.sms = sms > 0 ? sms : 148;
    c.ctx = current_context();  // the lookup above makes the primary context current
  }
  return &c;
}

unsigned int* device_status_word() {
  DeviceCache* c = dev_cache();
  return c ? c->status : nullptr;
}

int num_sms() {
  DeviceCache* c = dev_cache();
  return c ? c->sms : 148;
}

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

ndiff_status make_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                            const uint64_t* strides_bytes, const uint32_t* box) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return set_error(NDIFF_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  cuuint64_t gd[5];
  cuuint64_t gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) gs[i] = strides_bytes[i];
  }
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base),
                  gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(NDIFF_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
  return NDIFF_OK;
}

}  // namespace ndiff

using namespace ndiff;

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

extern "C" {

const char* ndiff_last_error(void) { return g_last_error; }

const char* ndiff_status_string(ndiff_status s) {
  switch (s) {
    case NDIFF_OK: return "NDIFF_OK";
    case NDIFF_ERR_INVALID_ARG: return "NDIFF_ERR_INVALID_ARG";
    case NDIFF_ERR_UNSUPPORTED: return "NDIFF_ERR_UNSUPPORTED";
    case NDIFF_ERR_CUDA: return "NDIFF_ERR_CUDA";
    case NDIFF_ERR_OOM: return "NDIFF_ERR_OOM";
    case NDIFF_ERR_WORKSPACE: return "NDIFF_ERR_WORKSPACE";
    case NDIFF_ERR_TIMEOUT: return "NDIFF_ERR_TIMEOUT";
  }
  return "unknown ndiff_status";
}

ndiff_status ndiff_check(cudaStream_t stream) {
  NDIFF_CUDA_TRY(cudaStreamSynchronize(stream));
  unsigned int* w = device_status_word();
  if (!w) return set_error(NDIFF_ERR_CUDA, "device status word unavailable");
  unsigned int v = 0;
  NDIFF_CUDA_TRY(cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost));
  if (v) {
    unsigned int z = 0;
    NDIFF_CUDA_TRY(cudaMemcpy(w, &z, sizeof(z), cudaMemcpyHostToDevice));
    if (v & kStatusTimeout)
      return set_error(NDIFF_ERR_TIMEOUT, "a bounded device wait expired (status 0x%x)", v);
    if (v & kStatusBadInput)
      return set_error(NDIFF_ERR_INVALID_ARG,
                       "a kernel read an input outside its range: kv_len outside [0, Lmax - T] or "
                       "a token id outside [0, V) (status 0x%x)",
                       v);
  }
  return NDIFF_OK;
}

namespace {
// One warp waits on a barrier that expects an arrival nothing makes; the wait
// gives up after limit_ns of %globaltimer, records the timeout and returns.
__global__ void selftest_timeout_kernel(unsigned long long limit_ns, unsigned int* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t b = smem_u32(&bar);
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait(b, 0)) {
      if (globaltimer() - t0 > limit_ns) {
        atomicOr(status, kStatusTimeout);
        break;
      }
    }
  }
  __syncthreads();
}
}  // namespace

extern "C++" {
namespace ndiff {
ndiff_status check_block_attn_args(ndiff_dtype dt, const void* q, const void* k, const void* v,
                                   const int32_t* kv_len, int B, int T, int Hq, int Hkv, int D,
                                   int Lmax, ndiff_mask mode, const void* out) {
  if (dt != NDIFF_BF16 && dt != NDIFF_F32)
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_block_attn: bad dtype %d", (int)dt);
  if (mode != NDIFF_BIDIR && mode != NDIFF_CAUSAL)
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_block_attn: bad mask mode %d", (int)mode);
  if (B < 0 || T < 1 || Hq < 1 || Hkv < 1 || D < 1 || Lmax < T)
    return set_error(NDIFF_ERR_INVALID_ARG,
                     "ndiff_block_attn: need B>=0, T>=1, heads>=1, D>=1, Lmax>=T (got B=%d T=%d "
                     "Hq=%d Hkv=%d D=%d Lmax=%d)",
                     B, T, Hq, Hkv, D, Lmax);
  if (Hq % Hkv != 0)
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_block_attn: Hq %% Hkv != 0 (%d, %d)", Hq, Hkv);
  if (B > 0 && (!q || !k || !v || !kv_len || !out))
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_block_attn: null pointer");
  if (dt == NDIFF_BF16) {
    if (D != 128)
      return set_error(NDIFF_ERR_UNSUPPORTED, "ndiff_block_attn: bf16 path needs D == 128 (got %d)", D);
    if ((Hq / Hkv) * T > 128)
      return set_error(NDIFF_ERR_UNSUPPORTED,
                       "ndiff_block_attn: bf16 path needs (Hq/Hkv)*T <= 128 (got %d)", (Hq / Hkv) * T);
    if ((long long)B * Hkv * Lmax >= (1LL << 31) || (long long)B * T >= (1LL << 31) || B > 65535)
      return set_error(NDIFF_ERR_UNSUPPORTED, "ndiff_block_attn: cache too large");
    if (B > 0 && (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)))
      return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_block_attn: bf16 pointers must be 16-byte aligned");
  } else {
    if (D > 64)
      return set_error(NDIFF_ERR_UNSUPPORTED, "ndiff_block_attn: f32 path needs D <= 64 (got %d)", D);
  }
  return NDIFF_OK;
}
}  // namespace ndiff
}  // extern "C++"

size_t ndiff_block_attn_split_workspace_size(ndiff_dtype dt, int B, int T, int Hq, int Hkv, int D,
                                             int Lmax, int split_keys) {
  if (dt != NDIFF_BF16 || B <= 0 || Hkv <= 0 || Lmax <= 0 || D != 128) return 0;
  const int split = split_keys > 0 ? split_keys : attn_bf16_auto_split(B, Hkv, Lmax);
  return attn_bf16_workspace(B, T, Hq, Hkv, Lmax, split);
}

size_t ndiff_block_attn_workspace_size(ndiff_dtype dt, int B, int T, int Hq, int Hkv, int D,
                                       int Lmax) {
  return ndiff_block_attn_split_workspace_size(dt, B, T, Hq, Hkv, D, Lmax, 0);
}

ndiff_status ndiff_block_attn_split(ndiff_dtype dt, const void* q, const void* k_cache,
                                    const void* v_cache, const int32_t* kv_len, int B, int T,
                                    int Hq, int Hkv, int D, int Lmax, ndiff_mask mode,
                                    float scale, int split_keys, void* out, void* ws,
                                    size_t ws_bytes, cudaStream_t stream) {
  ndiff_status s = check_block_attn_args(dt, q, k_cache, v_cache, kv_len, B, T, Hq, Hkv, D, Lmax, mode, out);
  if (s != NDIFF_OK) return s;
  if (split_keys < 0 || split_keys % 64 != 0)
    return set_error(NDIFF_ERR_INVALID_ARG,
                     "ndiff_block_attn: split_keys must be 0 or a positive multiple of 64 (got %d)",
                     split_keys);
  if (B == 0) return NDIFF_OK;
  const int causal = mode == NDIFF_CAUSAL ? 1 : 0;
  if (dt == NDIFF_F32)
    return launch_attn_f32(static_cast<const float*>(q), static_cast<const float*>(k_cache),
                           static_cast<const float*>(v_cache), kv_len, B, T, Hq, Hkv, D, Lmax,
                           causal, scale, static_cast<float*>(out), stream);
  const int split = split_keys > 0 ? split_keys : attn_bf16_auto_split(B, Hkv, Lmax);
  return launch_attn_bf16(q, k_cache, v_cache, kv_len, B, T, Hq, Hkv, Lmax, causal, scale, split,
                          out, ws, ws_bytes, stream);
}

ndiff_status ndiff_block_attn(ndiff_dtype dt, const void* q, const void* k_cache,
                              const void* v_cache, const int32_t* kv_len, int B, int T, int Hq,
                              int Hkv, int D, int Lmax, ndiff_mask mode, float scale, void* out,
                              void* ws, size_t ws_bytes, cudaStream_t stream) {
  return ndiff_block_attn_split(dt, q, k_cache, v_cache, kv_len, B, T, Hq, Hkv, D, Lmax, mode,
                                scale, 0, out, ws, ws_bytes, stream);
}

ndiff_status ndiff_logits_reduce(ndiff_dtype dt, const void* logits, int R, int V, int64_t ld,
                                 int exclude_id, int32_t* argmax, float* conf,
                                 cudaStream_t stream) {
  if (dt != NDIFF_BF16 && dt != NDIFF_F32)
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_logits_reduce: bad dtype %d", (int)dt);
  if (R < 0 || V < 1 || ld < V)
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_logits_reduce: need R>=0, V>=1, ld>=V (R=%d V=%d ld=%lld)",
                     R, V, (long long)ld);
  if (R == 0) return NDIFF_OK;
  if (!logits || !argmax || !conf)
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_logits_reduce: null pointer");
  if (!aligned16(logits) || (dt == NDIFF_BF16 ? ld % 8 : ld % 4) != 0)
    return set_error(NDIFF_ERR_INVALID_ARG,
                     "ndiff_logits_reduce: rows must start 16-byte aligned (pointer and ld)");
  return launch_logits_reduce(dt, logits, R, V, ld, exclude_id, argmax, conf, stream);
}

ndiff_status ndiff_unmask(const float* conf, const int32_t* pred, int B, int T, int k,
                          uint32_t* mask_bits, int32_t* block_in, int32_t* draft, int32_t* chosen,
                          cudaStream_t stream) {
  if (B < 0 || T < 1 || T > 32 || k < 1 || k > T)
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_unmask: need B>=0, 1<=T<=32, 1<=k<=T (B=%d T=%d k=%d)",
                     B, T, k);
  if (B == 0) return NDIFF_OK;
  if (!conf || !pred || !mask_bits || !block_in || !draft || !chosen)
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_unmask: null pointer");
  return launch_unmask(conf, pred, B, T, k, mask_bits, block_in, draft, chosen, stream);
}

ndiff_status ndiff_unmask_threshold(const float* conf, const int32_t* pred, int B, int T, float tau,
                                    float tau_revise, uint32_t* mask_bits, int32_t* block_in,
                                    int32_t* draft, int32_t* n_fixed, int32_t* n_revised,
                                    cudaStream_t stream) {
  if (B < 0 || T < 1 || T > 32 || !(tau >= 0.f) || !(tau_revise >= 0.f))
    return set_error(NDIFF_ERR_INVALID_ARG,
                     "ndiff_unmask_threshold: need B>=0, 1<=T<=32, tau>=0, tau_revise>=0 "
                     "(B=%d T=%d tau=%g tau_revise=%g)",
                     B, T, (double)tau, (double)tau_revise);
  if (B == 0) return NDIFF_OK;
  if (!conf || !pred || !mask_bits || !block_in || !draft)
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_unmask_threshold: null pointer");
  return launch_unmask_threshold(conf, pred, B, T, tau, tau_revise, mask_bits, block_in, draft,
                                 n_fixed, n_revised, stream);
}

ndiff_status ndiff_verify_accept(const int32_t* draft, const int32_t* target, int B, int T,
                                 int32_t* accept_len, int32_t* commit, int32_t* n_commit,
                                 int32_t* kv_len, cudaStream_t stream) {
  if (B < 0 || T < 1 || T > 32)
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_verify_accept: need B>=0, 1<=T<=32 (B=%d T=%d)", B, T);
  if (B == 0) return NDIFF_OK;
  if (!draft || !target || !accept_len || !commit || !n_commit)
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_verify_accept: null pointer");
  return launch_verify_accept(draft, target, B, T, accept_len, commit, n_commit, kv_len, stream);
}

ndiff_status ndiff_selftest_timeout(int limit_us, cudaStream_t stream) {
  if (limit_us < 1 || limit_us > 2000000)
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_selftest_timeout: limit_us in [1, 2000000] (got %d)",
                     limit_us);
  unsigned int* w = device_status_word();
  if (!w) return set_error(NDIFF_ERR_CUDA, "device status word unavailable");
  selftest_timeout_kernel<<<1, 32, 0, stream>>>((unsigned long long)limit_us * 1000ull, w);
  NDIFF_CUDA_TRY(cudaGetLastError());
  return NDIFF_OK;
}

size_t ndiff_gemm_bf16_workspace_size(int M, int N, int K) {
  if (M < 1 || N < 1 || K < 64) return 0;
  if (M > 32) return 0;  // the wide kernel needs no scratch
  const GemmPlan pl = gemm_plan(N, K);
  const size_t cnt = (((size_t)pl.ntiles * 4) + 255) & ~(size_t)255;
  return cnt + gemm_partials_bytes(pl);
}

ndiff_status ndiff_gemm_bf16(const void* x, const void* w, int M, int N, int K, float* y,
                             int64_t ldy, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (M < 1 || N < 1 || K < 64 || K % 64 != 0 || ldy < N)
    return set_error(NDIFF_ERR_INVALID_ARG,
                     "ndiff_gemm_bf16: need M>=1, N>=1, K a positive multiple of 64, ldy>=N "
                     "(M=%d N=%d K=%d ldy=%lld)",
                     M, N, K, (long long)ldy);
  if (!x || !w || !y) return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_gemm_bf16: null pointer");
  if (!aligned16(x) || !aligned16(w))
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_gemm_bf16: x and w must be 16-byte aligned");
  const size_t need = ndiff_gemm_bf16_workspace_size(M, N, K);
  if (need > 0 && (!ws || ws_bytes < need))
    return set_error(NDIFF_ERR_WORKSPACE, "ndiff_gemm_bf16: workspace of %zu bytes needed, %zu given",
                     need, ws_bytes);
  GemmParams p;
  memset(&p, 0, sizeof(p));
  p.N = N;
  p.T = M;
  p.mode = GEMM_EPI_F32;
  p.out = y;
  p.ldo = ldy;
  CUtensorMap tw, tx;
  if (M > 32) {
    ndiff_status s = gemm_make_maps(w, N, K, false, nullptr, 0, &tw, nullptr);
    if (s != NDIFF_OK) return s;
    s = gemm_wide_make_xmap(x, M, K, &tx, gemm_wide_box_rows(M));
    if (s != NDIFF_OK) return s;
    return launch_gemm_wide(tw, tx, gemm_wide_plan(N, K, M), p, stream);
  }
  const GemmPlan pl = gemm_plan(N, K);
  const size_t cnt = (((size_t)pl.ntiles * 4) + 255) & ~(size_t)255;
  ndiff_status s = gemm_make_maps(w, N, K, false, x, M, &tw, &tx);
  if (s != NDIFF_OK) return s;
  NDIFF_CUDA_TRY(cudaMemsetAsync(ws, 0, (size_t)pl.ntiles * 4, stream));
  p.counters = static_cast<int*>(ws);
  p.ws = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + cnt);
  return launch_gemm_bf16(tw, tx, pl, p, stream);
}

size_t ndiff_lm_head_argmax_workspace_size(int M, int N, int K) {
  if (M < 1 || N < 1 || K < 64) return 0;
  if (M > 32) {
    const GemmPlan pl = gemm_wide_plan(N, K, M);
    return (size_t)pl.ntiles * M * sizeof(float4);
  }
  const GemmPlan pl = gemm_plan(N, K);
  const size_t cnt = (((size_t)pl.ntiles * 4) + 255) & ~(size_t)255;
  const size_t part = (gemm_partials_bytes(pl) + 255) & ~(size_t)255;
  return cnt + part + (size_t)pl.ntiles * 32 * sizeof(float4);
}

ndiff_status ndiff_lm_head_argmax(const void* x, const void* w, int M, int N, int K, int exclude_id,
                                  int32_t* argmax, float* conf, void* ws, size_t ws_bytes,
                                  cudaStream_t stream) {
  if (M < 1 || N < 1 || K < 64 || K % 64 != 0 || exclude_id < -1 || exclude_id >= N)
    return set_error(NDIFF_ERR_INVALID_ARG,
                     "ndiff_lm_head_argmax: need M>=1, N>=1, K a positive multiple of 64, "
                     "-1<=exclude_id<N (M=%d N=%d K=%d exclude_id=%d)",
                     M, N, K, exclude_id);
  if (!x || !w || !argmax || !conf)
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_lm_head_argmax: null pointer");
  if (!aligned16(x) || !aligned16(w))
    return set_error(NDIFF_ERR_INVALID_ARG, "ndiff_lm_head_argmax: x and w must be 16-byte aligned");
  const size_t need = ndiff_lm_head_argmax_workspace_size(M, N, K);
  if (!ws || ws_bytes < need)
    return set_error(NDIFF_ERR_WORKSPACE,
                     "ndiff_lm_head_argmax: workspace of %zu bytes needed, %zu given", need, ws_bytes);
  GemmParams p;
  memset(&p, 0, sizeof(p));
  p.N = N;
  p.T = M;
  p.mode = GEMM_EPI_ARGMAX;
  p.excl = exclude_id;
  CUtensorMap tw, tx;
  if (M > 32) {
    const GemmPlan pl = gemm_wide_plan(N, K, M);
    ndiff_status s = gemm_make_maps(w, N, K, false, nullptr, 0, &tw, nullptr);
    if (s != NDIFF_OK) return s;
    s = gemm_wide_make_xmap(x, M, K, &tx, gemm_wide_box_rows(M));
    if (s != NDIFF_OK) return s;
    p.red = static_cast<float4*>(ws);
    s = launch_gemm_wide(tw, tx, pl, p, stream);
    if (s != NDIFF_OK) return s;
    return launch_argmax_merge(p.red, pl.ntiles, M, M, argmax, conf, stream);
  }
  const GemmPlan pl = gemm_plan(N, K);
  const size_t cnt = (((size_t)pl.ntiles * 4) + 255) & ~(size_t)255;
  const size_t part = (gemm_partials_bytes(pl) + 255) & ~(size_t)255;
  ndiff_status s = gemm_make_maps(w, N, K, false, x, M, &tw, &tx);
  if (s != NDIFF_OK) return s;
  NDIFF_CUDA_TRY(cudaMemsetAsync(ws, 0, (size_t)pl.ntiles * 4, stream));
  p.counters = static_cast<int*>(ws);
  p.ws = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + cnt);
  p.red = reinterpret_cast<float4*>(static_cast<uint8_t*>(ws) + cnt + part);
  s = launch_gemm_bf16(tw, tx, pl, p, stream);
  if (s != NDIFF_OK) return s;
  return launch_argmax_merge(p.red, pl.ntiles, M, 32, argmax, conf, stream);
}

}  // extern "C"
