// model.cu — placeholder for the model entry points (filled in below).
#include "common.cuh"
#include "kernels.h"

using namespace ndiff;

extern "C" {
ndiff_status ndiff_model_create(const ndiff_model_config*, uint64_t, ndiff_model**) {
  return set_error(NDIFF_ERR_UNSUPPORTED, "model not built yet");
}
ndiff_status ndiff_model_destroy(ndiff_model*) { return NDIFF_OK; }
ndiff_status ndiff_prefill(ndiff_model*, const int32_t*, int, cudaStream_t) {
  return set_error(NDIFF_ERR_UNSUPPORTED, "model not built yet");
}
ndiff_status ndiff_decode_step(ndiff_model*, ndiff_mode, int, int32_t*, int*, ndiff_stats*,
                               cudaStream_t) {
  return set_error(NDIFF_ERR_UNSUPPORTED, "model not built yet");
}
ndiff_status ndiff_model_forward(ndiff_model*, const int32_t*, int, ndiff_mask, float*,
                                 cudaStream_t) {
  return set_error(NDIFF_ERR_UNSUPPORTED, "model not built yet");
}
ndiff_status ndiff_model_state(const ndiff_model*, int*, int32_t*) {
  return set_error(NDIFF_ERR_UNSUPPORTED, "model not built yet");
}
ndiff_status ndiff_model_read_weight(const ndiff_model*, int, int64_t, int64_t, float*) {
  return set_error(NDIFF_ERR_UNSUPPORTED, "model not built yet");
}
}
