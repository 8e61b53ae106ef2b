// attn_noalloc.cu — block attention for callers that cannot allocate device
// memory.
//
// The split-KV bf16 attention needs scratch for its per-split partial results.
// ndiff_block_attn takes that scratch from the caller. Some callers cannot
// provide it: plugin interfaces that hand a kernel only its input and output
// buffers, and processes whose memory manager reserved the device memory up
// front so that a cudaMalloc would fail or would have to bypass the manager.
// ndiff_block_attn_noalloc serves them with a scratch array that lives in the
// library's own device image (kNoallocScratchBytes per GPU, held from the time
// the library is loaded on that GPU until the process exits). It performs no
// allocation of any kind.
//
// Set-up: the device address of the array is looked up by the first call made
// while a device is current, and again whenever the current CUDA context is no
// longer the one it was taken in (after a cudaDeviceReset, or under a context
// the caller made current); that first call should come before any stream
// capture. Every call shares the one array, so calls whose kernels overlap on
// the GPU (for instance on two streams) race on it and must be serialised by
// the caller. The array keeps whatever the last call left in it; nothing needs
// to start at zero, because every partial result the merge step reads was
// written earlier by the same call.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t kNoallocScratchBytes = NDIFF_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

struct ScratchAddr {
  void* ctx = nullptr;   // context the address was looked up in
  void* ptr = nullptr;
};
ScratchAddr g_scratch[64];
std::mutex g_scratch_mu;

// Device address of g_noalloc_scratch in the current context (host code must
// not pass the symbol itself to a kernel: on the host it names a stand-in).
ndiff_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return ndiff::cuda_error(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64)
    return ndiff::set_error(NDIFF_ERR_UNSUPPORTED, "ndiff_block_attn_noalloc: device %d", dev);
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  ScratchAddr& a = g_scratch[dev];
  void* ctx = ndiff::current_context();
  if (a.ptr == nullptr || ctx == nullptr || ctx != a.ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
      a.ptr = nullptr;
      return ndiff::cuda_error(e, "cudaGetSymbolAddress(scratch)");
    }
    a.ptr = p;
    a.ctx = ndiff::current_context();
  }
  *out = a.ptr;
  return NDIFF_OK;
}

}  // namespace

extern "C" ndiff_status ndiff_block_attn_noalloc(ndiff_dtype dt, const void* q,
                                                 const void* k_cache, const void* v_cache,
                                                 const int32_t* kv_len, int B, int T, int Hq,
                                                 int Hkv, int D, int Lmax, ndiff_mask mode,
                                                 float scale, void* out, cudaStream_t stream) {
  // the same argument errors as ndiff_block_attn, reported before the size check
  ndiff_status s = ndiff::check_block_attn_args(dt, q, k_cache, v_cache, kv_len, B, T, Hq, Hkv, D,
                                                Lmax, mode, out);
  if (s != NDIFF_OK) return s;
  const size_t need = ndiff_block_attn_workspace_size(dt, B, T, Hq, Hkv, D, Lmax);
  if (need > kNoallocScratchBytes)
    return ndiff::set_error(NDIFF_ERR_WORKSPACE,
                            "ndiff_block_attn_noalloc: this shape needs %zu bytes of scratch, "
                            "more than the built-in %zu; use ndiff_block_attn with a workspace",
                            need, kNoallocScratchBytes);
  void* ws = nullptr;
  if (need > 0) {
    s = scratch_address(&ws);
    if (s != NDIFF_OK) return s;
  }
  return ndiff_block_attn(dt, q, k_cache, v_cache, kv_len, B, T, Hq, Hkv, D, Lmax, mode, scale,
                          out, ws, need, stream);
}
