// sdv_hold.cuh -- a CTA's whole slice of one position (target row, and the
// draft row when there is one) brought into shared memory at once and kept
// there until the next position starts, so that the draw after a rejection
// (or the bonus draw) works on the same bytes instead of reading them again.
//
// The slice is cut in chunks of kStg vectors per row; chunk c lands in
// stage c (two rows of kStg vectors side by side, the layout of the ring in
// sdv_ring.cuh), every chunk with its own mbarrier.  Thread 0 issues every
// chunk of the pass at once, so a CTA has its whole slice in flight; the
// threads consume the chunks in order as they land.  Each wait is bounded
// (mbar_wait reports SD_DEV_TIMEOUT and returns).
#pragma once

#include "sdv_device.cuh"
#include "sdv_ring.cuh"
#include "sdv_tma.cuh"

namespace sdv {

constexpr int kHoldMax = 16;  // chunks (stages) a held slice may take

struct Hold {
  uint4 *buf;        // [kHoldMax][kStageVecs], as many as the slice needs
  uint64_t *full;    // [kHoldMax] mbarriers: chunk landed (tx bytes)
  uint32_t phase;    // bit c: parity of chunk c's next completion
  int32_t *dev_status;
};

// Every thread calls it (it holds a block barrier).
__device__ __forceinline__ void hold_init(Hold &h) {
  if (threadIdx.x == 0) {
    for (int c = 0; c < kHoldMax; ++c) mbar_init(&h.full[c], 1);
    fence_mbar_init();
  }
  h.phase = 0;
  __syncthreads();
}

// Chunks of a slice of nv vectors.
__device__ __forceinline__ int hold_chunks(const Slice &sl) {
  return (sl.vend - sl.vbeg + kStg - 1) / kStg;
}

// Online softmax states of row A (and B when non-null) over the slice,
// leaving the slice in shared memory.  Every thread calls it; the block
// barrier at the start keeps the copies from overwriting chunks that a
// thread still reads from the previous pass.
template <int DT, int VW>
__device__ __forceinline__ void hold_stats(Hold &h, const char *rowA,
                                           const char *rowB, const Slice &sl,
                                           float k2, MS &a, MS &b) {
  const int nv = sl.vend - sl.vbeg;
  const int nch = hold_chunks(sl);
  __syncthreads();
  if (threadIdx.x == 0) {
    fence_proxy_async();
    for (int c = 0; c < nch; ++c) {
      const int v0 = c * kStg;
      const uint32_t bytes = (uint32_t)min(kStg, nv - v0) * 16u;
      mbar_expect_tx(&h.full[c], rowB ? 2u * bytes : bytes);
      bulk_g2s(h.buf + (size_t)c * kStageVecs,
               rowA + (size_t)(sl.vbeg + v0) * 16, bytes, &h.full[c]);
      if (rowB)
        bulk_g2s(h.buf + (size_t)c * kStageVecs + kStg,
                 rowB + (size_t)(sl.vbeg + v0) * 16, bytes, &h.full[c]);
    }
  }
  const bool hb = rowB != nullptr;
  for (int c = 0; c < nch; ++c) {
    mbar_wait(&h.full[c], (h.phase >> c) & 1u, h.dev_status);
    h.phase ^= 1u << c;
    const uint4 *A = h.buf + (size_t)c * kStageVecs;
    const int n = min(kStg, nv - c * kStg);
    for (int i = threadIdx.x; i < n; i += kThreads) {
      ms_add<DT, VW>(a, sget<DT, VW>(A, i), k2);
      if (hb) ms_add<DT, VW>(b, sget<DT, VW>(A + kStg, i), k2);
    }
  }
}

// Per-segment masses (segment s = vectors vbeg + 32 s ..) of the weights W
// over the slice that the last hold_stats left in shared memory (row B is
// read only when has_q); warp w takes segments w, w + 8, ... of each chunk,
// as ring_mass does.
template <int DT, int VW>
__device__ __forceinline__ void held_mass(const Hold &h, bool has_q,
                                          const Weight &W, const Slice &sl,
                                          float *segmass) {
  static_assert(kStg % 32 == 0, "whole segments per chunk");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nv = sl.vend - sl.vbeg;
  const int nch = hold_chunks(sl);
  for (int c = 0; c < nch; ++c) {
    const uint4 *A = h.buf + (size_t)c * kStageVecs;
    const uint4 *Bp = has_q ? A + kStg : A;
    const int n = min(kStg, nv - c * kStg);
    const int seg0 = c * (kStg / 32);
    for (int g = warp; g * 32 < n; g += kWarps) {  // warp-uniform
      const int i = g * 32 + lane;
      float acc = 0.f;
      if (i < n) {
        float w[VW];
        weights<DT, VW>(sget<DT, VW>(A, i), sget<DT, VW>(Bp, i), has_q, W, w);
#pragma unroll
        for (int e = 0; e < VW; ++e) acc += w[e];
      }
      acc = warp_down_sum(acc);
      if (lane == 0) segmass[seg0 + g] = acc;
    }
  }
}

}  // namespace sdv
