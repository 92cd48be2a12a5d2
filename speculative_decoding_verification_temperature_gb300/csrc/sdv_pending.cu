// sdv_pending.cu -- entry points declared in sd_verify.h whose kernels are
// not built yet: they reject every call with SD_ERR_UNSUPPORTED.
#include "sdv_host.cuh"

extern "C" size_t sd_verify_linear_fanout_workspace(int, int, int, sd_dtype) {
  return 256;
}
extern "C" sd_status sd_verify_linear_fanout(
    const void *, const void *, sd_dtype, const int32_t *, const float *, int,
    int, int, float, const int32_t *, int32_t *, int32_t *, float *,
    int32_t *, float *, int32_t *, void *, size_t, void *) {
  return sdv::fail(SD_ERR_UNSUPPORTED, "sd_verify_linear_fanout: not built");
}
