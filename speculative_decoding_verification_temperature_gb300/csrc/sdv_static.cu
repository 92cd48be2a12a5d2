// sdv_static.cu -- linear verify with its scratch in a file-scope device
// array instead of a caller-supplied workspace, for callers that must not
// allocate (the method itself has no such requirement).
//
// The array exists once per device.  Its address is looked up with
// cudaGetSymbolAddress (with the device current) on every call made outside
// a stream capture, so a device reset cannot leave a stale address behind;
// a call made while its stream is being captured reuses the address found
// by the last uncaptured call on that device (the first call on a device
// must therefore come before any capture).  Nothing is allocated or freed,
// here or in the path the array is handed to (sd_verify_linear, which
// clears the counters that must start at zero with a memset on the stream).
// Two calls whose work overlaps on the GPU share the array and race.
#include <mutex>

#include "sdv_host.cuh"

namespace sdv {

static __device__ __align__(256) unsigned char g_static_ws[SD_STATIC_WS_BYTES];

constexpr int kMaxDevices = 64;
static std::mutex g_static_mu;
static void *g_static_ptr[kMaxDevices];

static sd_status static_scratch(cudaStream_t stream, void **out) {
  int dev = 0;
  SDV_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices)
    return fail(SD_ERR_UNSUPPORTED, "device ordinal %d >= %d", dev,
                kMaxDevices);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  SDV_CUDA(cudaStreamIsCapturing(stream, &cap));
  std::lock_guard<std::mutex> g(g_static_mu);
  if (cap == cudaStreamCaptureStatusNone) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_ws);
    if (e != cudaSuccess)
      return fail(SD_ERR_CUDA, "cudaGetSymbolAddress of the static scratch: %s",
                  cudaGetErrorString(e));
    g_static_ptr[dev] = p;
  } else if (!g_static_ptr[dev]) {
    return fail(SD_ERR_INVALID_ARG,
                "first call on device %d inside a stream capture: make one "
                "call outside the capture first", dev);
  }
  *out = g_static_ptr[dev];
  return SD_OK;
}

}  // namespace sdv

extern "C" sd_status sd_verify_linear_static(
    const void *target_logits, const void *draft_logits, sd_dtype dt,
    const int32_t *draft_tokens, const float *uniforms, int B, int gamma,
    int V, float T, int32_t *n_accepted, int32_t *out_tokens, float *out_prob,
    float *out_accept_prob, float *out_resid, int32_t *dev_status,
    void *stream) {
  using namespace sdv;
  SDV_REQUIRE(dt == SD_F32 || dt == SD_BF16, "bad dtype %d", (int)dt);
  SDV_REQUIRE(B >= 0, "B < 0");
  SDV_REQUIRE(gamma >= 0 && gamma <= SD_MAX_GAMMA, "gamma=%d outside [0, %d]",
              gamma, SD_MAX_GAMMA);
  SDV_REQUIRE(V >= 1 && V <= SD_MAX_V, "V=%d outside [1, %d]", V, SD_MAX_V);
  if (B == 0) return SD_OK;
  const size_t need = sd_verify_linear_workspace(B, gamma, V, dt);
  if (need > (size_t)SD_STATIC_WS_BYTES)
    return fail(SD_ERR_UNSUPPORTED,
                "B=%d gamma=%d V=%d needs %zu B of scratch, above the static "
                "%zu B (SD_STATIC_WS_BYTES): use sd_verify_linear with a "
                "workspace",
                B, gamma, V, need, (size_t)SD_STATIC_WS_BYTES);
  int sms = 0;
  const sd_status dst = check_device(&sms);  // SD_ERR_UNSUPPORTED off sm_103
  if (dst != SD_OK) return dst;
  void *ws = nullptr;
  const sd_status st = static_scratch(static_cast<cudaStream_t>(stream), &ws);
  if (st != SD_OK) return st;
  return sd_verify_linear(target_logits, draft_logits, dt, draft_tokens,
                          uniforms, B, gamma, V, T, n_accepted, out_tokens,
                          out_prob, out_accept_prob, out_resid, dev_status, ws,
                          (size_t)SD_STATIC_WS_BYTES, stream);
}
