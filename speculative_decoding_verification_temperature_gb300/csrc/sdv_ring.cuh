// sdv_ring.cuh -- streaming a CTA's slice of one or two rows through a ring
// of shared-memory stages filled by TMA bulk copies (cp.async.bulk with one
// mbarrier per stage).
//
// Thread 0 keeps kStages chunks in flight; every thread consumes chunk c
// as soon as its stage's "full" barrier completes, and the stage is refilled
// with chunk c + kStages after a block barrier (SDV_RING_SYNC=1, measured
// faster) or once every warp has arrived on the stage's "empty" barrier
// (SDV_RING_SYNC=0: warps then run ahead of each other by up to kStages - 1
// chunks).  The bytes in flight per CTA are the whole ring, independent of
// registers, so several CTAs per SM keep HBM busy while each one also
// spends time in cluster barriers.
#pragma once

#include "sdv_device.cuh"
#include "sdv_tma.cuh"

namespace sdv {

#ifndef SDV_STAGES
#define SDV_STAGES 3
#endif
#ifndef SDV_STG
#define SDV_STG 512
#endif
#ifndef SDV_RING_SYNC
#define SDV_RING_SYNC 1
#endif
constexpr int kStg = SDV_STG;         // 16-byte vectors per row per stage
constexpr int kStages = SDV_STAGES;   // stages in flight
constexpr int kStageVecs = 2 * kStg;  // a stage: two rows of kStg or one of 2 kStg
constexpr int kRingBytes = kStages * kStageVecs * 16;  // 48 KB

struct Ring {
  uint4 *buf;          // [kStages][kStageVecs]
  uint64_t *full;      // [kStages] mbarriers: data landed (tx bytes)
  uint64_t *empty;     // [kStages] mbarriers: every warp is done with it
  uint32_t phase;      // bit s: parity of stage s's next "full" completion
  uint32_t used;       // thread 0: bit s set once stage s was filled
  uint32_t epar;       // thread 0: bit s: parity of the "empty" wait due
  int32_t *dev_status;
  uint64_t policy;     // L2 cache policy of the copies (0: the default)
};

__device__ __forceinline__ void ring_init(Ring &rg) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&rg.full[s], 1);
      mbar_init(&rg.empty[s], kWarps);
    }
    fence_mbar_init();
  }
  rg.phase = 0;
  rg.used = 0;
  rg.epar = 0;
  rg.policy = 0;
  __syncthreads();
}

// One pass over this CTA's slice of row A (and row B when non-null), in
// chunks of STG vectors: kStg for two rows, up to 2 kStg for row A alone.
// f(a, b, v0, n) is called by every thread for each chunk: a / b point at
// the chunk's n vectors in shared memory, v0 is the absolute index of the
// chunk's first vector.  Block-uniform control flow is required.
template <int STG = kStg, class F>
__device__ __forceinline__ void ring_pass(Ring &rg, const char *rowA,
                                          const char *rowB, const Slice &sl,
                                          F &&f) {
  static_assert(STG == kStg || STG == kStageVecs, "chunk of one stage");
  const int nv = sl.vend - sl.vbeg;
  const int nch = (nv + STG - 1) / STG;
  auto issue = [&](int c) {  // thread 0 only
    const int s = c % kStages;
    const int v0 = c * STG;
    const int cnt = min(STG, nv - v0);
    const uint32_t bytes = (uint32_t)cnt * 16u;
    if (!SDV_RING_SYNC && (rg.used >> s & 1u)) {  // every warp released it
      mbar_wait(&rg.empty[s], (rg.epar >> s) & 1u, rg.dev_status);
      rg.epar ^= 1u << s;
    }
    rg.used |= 1u << s;
    fence_proxy_async();
    mbar_expect_tx(&rg.full[s], bytes * ((STG == kStg && rowB) ? 2u : 1u));
    if (rg.policy) {
      bulk_g2s_hint(rg.buf + (size_t)s * kStageVecs,
                    rowA + (size_t)(sl.vbeg + v0) * 16, bytes, &rg.full[s],
                    rg.policy);
      if (STG == kStg && rowB)
        bulk_g2s_hint(rg.buf + (size_t)s * kStageVecs + kStg,
                      rowB + (size_t)(sl.vbeg + v0) * 16, bytes, &rg.full[s],
                      rg.policy);
    } else {
      bulk_g2s(rg.buf + (size_t)s * kStageVecs,
               rowA + (size_t)(sl.vbeg + v0) * 16, bytes, &rg.full[s]);
      if (STG == kStg && rowB)
        bulk_g2s(rg.buf + (size_t)s * kStageVecs + kStg,
                 rowB + (size_t)(sl.vbeg + v0) * 16, bytes, &rg.full[s]);
    }
  };
  if (threadIdx.x == 0)
    for (int c = 0; c < nch && c < kStages; ++c) issue(c);
  for (int c = 0; c < nch; ++c) {
    const int s = c % kStages;
    mbar_wait(&rg.full[s], (rg.phase >> s) & 1u, rg.dev_status);
    rg.phase ^= 1u << s;
    f(rg.buf + (size_t)s * kStageVecs, rg.buf + (size_t)s * kStageVecs + kStg,
      sl.vbeg + c * STG, min(STG, nv - c * STG));
#if SDV_RING_SYNC
    __syncthreads();
    if (threadIdx.x == 0 && c + kStages < nch) issue(c + kStages);
#else
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&rg.empty[s]);
    if (threadIdx.x == 0 && c + kStages < nch) issue(c + kStages);
#endif
  }
}

template <int DT, int VW>
__device__ __forceinline__ Raw<DT, VW> sget(const uint4 *p, int i) {
  Raw<DT, VW> r;
  r.w = p[i];
  return r;
}

// Online softmax states of row A (and B) over the slice.
template <int DT, int VW>
__device__ __forceinline__ void ring_stats(Ring &rg, const char *rowA,
                                           const char *rowB, const Slice &sl,
                                           float k2, MS &a, MS &b) {
  const bool hb = rowB != nullptr;
  ring_pass(rg, rowA, rowB, sl, [&](const uint4 *A, const uint4 *Bp, int,
                                    int n) {
    for (int i = threadIdx.x; i < n; i += kThreads) {
      ms_add<DT, VW>(a, sget<DT, VW>(A, i), k2);
      if (hb) ms_add<DT, VW>(b, sget<DT, VW>(Bp, i), k2);
    }
  });
}

// Greedy argmax state of row A over the slice.
template <int DT, int VW>
__device__ __forceinline__ void ring_argmax(Ring &rg, const char *rowA,
                                            const Slice &sl, AM &a) {
  ring_pass(rg, rowA, nullptr, sl, [&](const uint4 *A, const uint4 *, int v0,
                                       int n) {
    for (int i = threadIdx.x; i < n; i += kThreads)
      am_add<DT, VW>(a, sget<DT, VW>(A, i), (v0 + i) * VW);
  });
}

// Per-segment masses (segment s = vectors vbeg + 32 s ..) of the weights
// W over the slice; a chunk holds kStg / 32 segments, warp w takes
// segments w, w + 8, ...
template <int DT, int VW>
__device__ __forceinline__ void ring_mass(Ring &rg, const char *rowA,
                                          const char *rowB, bool has_q,
                                          const Weight &W, const Slice &sl,
                                          float *segmass) {
  static_assert(kStg % 32 == 0, "whole segments per chunk");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  ring_pass(rg, rowA, has_q ? rowB : nullptr, sl,
            [&](const uint4 *A, const uint4 *Bp, int v0, int n) {
              const int seg0 = (v0 - sl.vbeg) / 32;
              for (int g = warp; g * 32 < n; g += kWarps) {  // warp-uniform
                const int i = g * 32 + lane;
                float acc = 0.f;
                if (i < n) {
                  float w[VW];
                  weights<DT, VW>(sget<DT, VW>(A, i),
                                  sget<DT, VW>(has_q ? Bp : A, i), has_q, W,
                                  w);
#pragma unroll
                  for (int e = 0; e < VW; ++e) acc += w[e];
                }
                acc = warp_down_sum(acc);
                if (lane == 0) segmass[seg0 + g] = acc;
              }
            });
}

}  // namespace sdv
