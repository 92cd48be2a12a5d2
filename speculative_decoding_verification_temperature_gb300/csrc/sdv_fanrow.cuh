// sdv_fanrow.cuh -- the fan-out's exact top-F of one draft row (Speculative
// Speculative Decoding / Saguaro, "speculation cache strategy") by a single
// CTA through the TMA ring, and the block-wide ranking of key lists that
// both the fan-out kernel and the verify fused with it use.
#pragma once

#include "sdv_ring.cuh"
#include "sdv_topf.cuh"

namespace sdv {

// One row slice through the warp filters, via the TMA ring in chunks of
// kStageVecs vectors: warp w takes vectors 32 w .. 32 w + 31,
// 32 (w + kWarps) .., ... of every chunk.
template <int DT, int VW>
__device__ __forceinline__ void filter_pass_ring(Ring &rg, const char *row,
                                                 const Slice &sl,
                                                 WarpFilter &w,
                                                 uint32_t *cta_th) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  ring_pass<kStageVecs>(rg, row, nullptr, sl, [&](const uint4 *A,
                                                  const uint4 *, int v0,
                                                  int n) {
    wf_sync(w, cta_th);
    if (n == kStageVecs) {  // full chunk: no idle lanes
#pragma unroll 2
      for (int base = warp * 32; base < kStageVecs; base += kThreads) {
        const int i = base + lane;
        wf_offer<DT, VW>(w, cta_th, sget<DT, VW>(A, i), true, (v0 + i) * VW);
      }
    } else {
      for (int base = warp * 32; base < n; base += kThreads) {  // warp-uniform
        const int i = base + lane;
        Raw<DT, VW> r{};
        if (i < n) r = sget<DT, VW>(A, i);
        wf_offer<DT, VW>(w, cta_th, r, i < n, (v0 + i) * VW);
      }
    }
  });
}

// Rank the keys in[0, C) (0 = empty; non-empty keys are unique) by counting
// and place the best F in out[] (descending).  Returns min(F, non-empty
// keys).  Block-wide; every thread gets the count.
__device__ __forceinline__ int rank_keys(const uint64_t *in, int C, int F,
                                         uint64_t *out) {
  int nz = 0;
  for (int i0 = 0; i0 < C; i0 += kThreads) {
    const int i = i0 + (int)threadIdx.x;
    const uint64_t me = i < C ? in[i] : 0;
    if (me != 0) {
      int rank = 0;
      for (int j = 0; j < C; ++j) rank += in[j] > me;
      if (rank < F) out[rank] = me;
    }
    nz += __syncthreads_count(me != 0);
  }
  __syncthreads();
  return nz < F ? nz : F;
}

// Write a row's top-F: token ids and logits of the first n keys, -1 / NaN
// for the rest, and for every slot when the row holds a NaN (status bit).
__device__ __forceinline__ void fan_write(const uint64_t *keys, int n, int F,
                                          bool nan, int32_t *otok,
                                          float *olog, int32_t *dev_status) {
  for (int i = threadIdx.x; i < F; i += kThreads) {
    const bool ok = !nan && i < n;
    otok[i] = ok ? key_idx(keys[i]) : -1;
    if (olog) olog[i] = ok ? key_val(keys[i]) : __int_as_float(0x7fc00000);
  }
  if (threadIdx.x == 0 && nan) status_or(dev_status, SD_DEV_NONFINITE);
}

// The exact top-F (F <= SD_MAX_FANOUT) of a whole row by this CTA alone.
// scratch holds kWarps * F keys and out F keys; *cta_th must be 0 on entry
// and is 0 again on return.  Block-wide.
template <int DT, int VW>
__device__ __forceinline__ void cta_row_topf(Ring &rg, uint32_t *cta_th,
                                             uint64_t *scratch, uint64_t *out,
                                             const char *row, int V, int F,
                                             int32_t *otok, float *olog,
                                             int32_t *dev_status) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const Slice sl = make_slice(V / VW, 0, 1);
  WarpFilter w;
  wf_init(w, F);
  filter_pass_ring<DT, VW>(rg, row, sl, w, cta_th);
  const bool nan = __syncthreads_or(w.nseen != w.nseen) != 0;
  if (lane < F) scratch[warp * F + lane] = w.a;
  if (32 + lane < F) scratch[warp * F + 32 + lane] = w.b;
  __syncthreads();
  const int n = rank_keys(scratch, kWarps * F, F, out);
  if (threadIdx.x == 0) *cta_th = 0;
  fan_write(out, n, F, nan, otok, olog, dev_status);
  __syncthreads();
}

}  // namespace sdv
