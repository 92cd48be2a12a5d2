// sdv_host.cu -- host helpers and the host-only entry points (version,
// last error, geometric fan-out schedule).
#include "sdv_host.cuh"

#include <atomic>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

namespace sdv {

namespace {
thread_local char g_err[256] = "";
std::mutex g_mu;

struct KeyHash {
  size_t operator()(const std::tuple<const void *, int, size_t, int> &k) const {
    return std::hash<const void *>()(std::get<0>(k)) ^
           (std::hash<int>()(std::get<1>(k)) << 1) ^
           (std::hash<size_t>()(std::get<2>(k)) << 7) ^
           (std::hash<int>()(std::get<3>(k)) << 13);
  }
};
std::unordered_map<std::tuple<const void *, int, size_t, int>, int, KeyHash>
    g_clusters;
std::unordered_map<int, int> g_dev_ok;  // device -> SM count (0: unsupported)
}  // namespace

sd_status fail(sd_status st, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return st;
}

namespace {
// defaults: the fastest measured configuration
std::atomic<int> g_tune[SD_TUNE_COUNT] = {
    {0},  // SD_TUNE_CLUSTER
    {0},  // SD_TUNE_NO_TMA
    {1},  // SD_TUNE_ALLROWS
    {1},  // SD_TUNE_SPEC
    {1},  // SD_TUNE_FUSED
    {1},  // SD_TUNE_KCAND_RING
    {0},  // SD_TUNE_FANOUT_CLUSTER
    {0},  // SD_TUNE_FANOUT_LDG
    {0},  // SD_TUNE_FANOUT_MAXC
    {1},  // SD_TUNE_FANOUT_L2_FIRST
    {1},  // SD_TUNE_HELPERS
};

bool tune_valid(int key, int v) {
  switch (key) {
    case SD_TUNE_CLUSTER:
    case SD_TUNE_FANOUT_CLUSTER:
      return v == 0 || v == 1 || v == 2 || v == 4 || v == 8 || v == 16;
    case SD_TUNE_ALLROWS:
    case SD_TUNE_SPEC:
      return v >= 0 && v <= 2;
    case SD_TUNE_FANOUT_MAXC:
      return v >= 0;
    default:
      return v == 0 || v == 1;
  }
}
}  // namespace

int tune(sd_tune key) {
  return (key >= 0 && key < SD_TUNE_COUNT)
             ? g_tune[key].load(std::memory_order_relaxed)
             : 0;
}

sd_status check_device(int *sm_count) {
  int dev = 0;
  SDV_CUDA(cudaGetDevice(&dev));
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_dev_ok.find(dev);
    if (it != g_dev_ok.end()) {
      if (!it->second)
        return fail(SD_ERR_UNSUPPORTED, "device %d is not sm_103", dev);
      *sm_count = it->second;
      return SD_OK;
    }
  }
  int major = 0, minor = 0, sms = 0;
  SDV_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor,
                                  dev));
  SDV_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor,
                                  dev));
  SDV_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const bool ok = (major == 10 && minor == 3);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    g_dev_ok[dev] = ok ? sms : 0;
  }
  if (!ok)
    return fail(SD_ERR_UNSUPPORTED, "device %d is sm_%d%d, not sm_103", dev,
                major, minor);
  *sm_count = sms;
  return SD_OK;
}

sd_status max_active_clusters(const void *kernel, int cl, size_t smem,
                              int *out) {
  int dev = 0;
  SDV_CUDA(cudaGetDevice(&dev));
  auto key = std::make_tuple(kernel, cl, smem, dev);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_clusters.find(key);
    if (it != g_clusters.end()) {
      *out = it->second;
      return SD_OK;
    }
  }
  if (cl > 8)
    SDV_CUDA(cudaFuncSetAttribute(
        kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1));
  {
    // allow every dynamic size the device can give next to the kernel's
    // static shared memory (the launch's own size sets the occupancy)
    cudaFuncAttributes fa;
    SDV_CUDA(cudaFuncGetAttributes(&fa, kernel));
    int optin = 0;
    SDV_CUDA(cudaDeviceGetAttribute(&optin,
                                    cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                    dev));
    const int room = optin - (int)fa.sharedSizeBytes;
    if ((long long)smem > room)
      return fail(SD_ERR_UNSUPPORTED, "%zu B of shared memory do not fit",
                  smem);
    SDV_CUDA(cudaFuncSetAttribute(
        kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, room));
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cl, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  SDV_CUDA(cudaOccupancyMaxActiveClusters(&n, kernel, &cfg));
  if (n <= 0)
    return fail(SD_ERR_UNSUPPORTED, "no cluster of %d CTAs fits (smem %zu)",
                cl, smem);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    g_clusters[key] = n;
  }
  *out = n;
  return SD_OK;
}

sd_status launch_clusters(const void *kernel, int nclusters, int cl,
                          size_t smem, cudaStream_t stream, void **args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(nclusters * cl), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  SDV_CUDA(cudaLaunchKernelExC(&cfg, kernel, args));
  return SD_OK;
}

sd_status launch_pdl(const void *kernel, unsigned grid, unsigned block,
                     size_t smem, cudaStream_t stream, void **args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(block, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  SDV_CUDA(cudaLaunchKernelExC(&cfg, kernel, args));
  return SD_OK;
}

}  // namespace sdv

extern "C" const char *sd_version(void) { return "sdverify 0.1 (sm_103a)"; }

extern "C" const char *sd_last_error(void) { return sdv::g_err; }

extern "C" sd_status sd_tune_set(sd_tune key, int value) {
  const int k = (int)key;
  SDV_REQUIRE(k >= 0 && k < SD_TUNE_COUNT, "unknown tuning key %d", k);
  SDV_REQUIRE(sdv::tune_valid(k, value), "value %d out of range for key %d",
              value, k);
  sdv::g_tune[k].store(value, std::memory_order_relaxed);
  return SD_OK;
}

extern "C" int sd_tune_get(sd_tune key) {
  const int k = (int)key;
  if (k < 0 || k >= SD_TUNE_COUNT) return -1;
  return sdv::g_tune[k].load(std::memory_order_relaxed);
}

// Saguaro, Theorem 12: w_k = a^{k/(1+r)} (k < K), w_K = a^{K/(1+r)}
// (1-a)^{-1/(1+r)}; F_k = F_0 w_k with F_0 = budget / sum w, made integer by
// handing the units left after flooring to the largest fractional parts
// (ties to the lower k).
extern "C" sd_status sd_fanout_schedule(int K, int budget, double a, double r,
                                        int32_t *F) {
  SDV_REQUIRE(F != nullptr, "F is null");
  SDV_REQUIRE(K >= 0 && K <= SD_MAX_K, "K=%d outside [0, %d]", K, SD_MAX_K);
  SDV_REQUIRE(budget >= 0, "budget < 0");
  SDV_REQUIRE(a > 0.0 && a < 1.0, "a must lie in (0, 1)");
  SDV_REQUIRE(r > 0.0 && std::isfinite(r), "r must be > 0");
  std::vector<double> w(K + 1), rem(K + 1);
  double total = 0.0;
  const double e = 1.0 / (1.0 + r);
  for (int k = 0; k <= K; ++k) {
    w[k] = std::pow(a, k * e);
    if (k == K) w[k] *= std::pow(1.0 - a, -e);
    total += w[k];
  }
  const double F0 = budget / total;
  int used = 0;
  for (int k = 0; k <= K; ++k) {
    const double x = F0 * w[k];
    const double fl = std::floor(x);
    F[k] = (int32_t)fl;
    rem[k] = x - fl;
    used += F[k];
  }
  for (int left = budget - used; left > 0; --left) {
    int best = -1;
    for (int k = 0; k <= K; ++k)
      if (rem[k] >= 0.0 && (best < 0 || rem[k] > rem[best])) best = k;
    if (best < 0) break;
    ++F[best];
    rem[best] = -1.0;
  }
  return SD_OK;
}
