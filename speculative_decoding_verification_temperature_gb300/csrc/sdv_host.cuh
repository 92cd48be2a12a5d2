// sdv_host.cuh -- host-side helpers shared by the entry points: argument
// checks with a thread-local error text, the sm_103 device check, cluster
// sizing and the cluster launch itself.
#pragma once

#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <unordered_map>

#include "sd_verify.h"

namespace sdv {

sd_status fail(sd_status st, const char *fmt, ...);
sd_status check_device(int *sm_count);
// Current value of a tuning switch (sd_tune_set); the defaults are the
// measured best.
int tune(sd_tune key);

#define SDV_REQUIRE(cond, ...)                              \
  do {                                                      \
    if (!(cond)) return ::sdv::fail(SD_ERR_INVALID_ARG, __VA_ARGS__); \
  } while (0)

#define SDV_CUDA(call)                                                   \
  do {                                                                   \
    cudaError_t e_ = (call);                                             \
    if (e_ != cudaSuccess)                                               \
      return ::sdv::fail(SD_ERR_CUDA, "%s: %s", #call,                   \
                         cudaGetErrorString(e_));                        \
  } while (0)

inline bool aligned16(const void *p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// Cluster size for rows of nvec vectors: slices of at least ~512 vectors
// (one load batch per thread), at most 16 CTAs.  SD_TUNE_CLUSTER overrides
// it (1, 2, 4, 8 or 16).
inline int choose_cluster(long long nvec) {
  int forced = tune(SD_TUNE_CLUSTER);
  if (forced == 1 || forced == 2 || forced == 4 || forced == 8 ||
      forced == 16)
    return forced;
  int cl = 1;
  while (cl < 16 && nvec / (2 * cl) >= 512) cl *= 2;
  return cl;
}

// Largest number of co-resident clusters of `cl` CTAs for a kernel (cached
// per kernel, cluster size and shared-memory size).
sd_status max_active_clusters(const void *kernel, int cl, size_t smem,
                              int *out);

// Launch `kernel` with a 1-D grid of nclusters * cl CTAs in clusters of cl.
sd_status launch_clusters(const void *kernel, int nclusters, int cl,
                          size_t smem, cudaStream_t stream, void **args);

// Launch `kernel` (1-D grid) with programmatic stream serialisation: it may
// start while the previous kernel in the stream is finishing, so it must
// wait (griddep_wait) before reading anything that kernel writes.
sd_status launch_pdl(const void *kernel, unsigned grid, unsigned block,
                     size_t smem, cudaStream_t stream, void **args);

// Row maps and output shape of a token tree whose nodes read rows of
// another tensor (sdv_trie.cu): node u of sequence b reads target row
// trow[b][u] of the sequence's trows rows and draft row drow[b][u] of its
// drows rows (-1: none); out_tokens has out_cols columns; out_cand[b]
// (nullable) gets node_cand[b][last accepted node], 0 when none.
struct TreeMaps {
  const int32_t *trow, *drow;
  int trows, drows;
  int out_cols;
  const int32_t *node_cand;
  int32_t *out_cand;
};

// The tree walk of sd_verify_tree (det = false) or sd_verify_tree_det
// (det = true), with optional row maps (sdv_tree.cu).
sd_status tree_launch(const void *target_logits, const void *draft_logits,
                      sd_dtype dt, const int32_t *parent,
                      const int32_t *node_tokens, const float *uniforms,
                      int B, int N, int V, float T, bool det,
                      int32_t *n_accepted, int32_t *out_tokens,
                      int32_t *out_nodes, float *out_prob,
                      int32_t *dev_status, void *workspace, size_t ws_bytes,
                      void *stream, const TreeMaps *maps = nullptr);

}  // namespace sdv
