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

// ------------------------------------------------------------------------
// Candidates of a row's top-F gathered while another pass streams it: each
// thread keeps the vector holding the largest element it has seen (16 raw
// bytes and the vector's index; an equal maximum later does not replace it)
// and the largest maximum among its other vectors, t2.  A vector costs two
// compares of its maximum, which the pass computes anyway.  The row's
// exact top-F follows from the kept vectors when every t2 lies strictly
// below the F-th best candidate's value: every element at or above that key
// is then in a kept vector.  A thread that met a NaN or an infinity stores
// t2 = +inf, so the check fails and the row is read whole.
template <int DT, int VW>
struct VecTop {
  Raw<DT, VW> best;
  int bidx;
  float t1, t2;
};

template <int DT, int VW>
__device__ __forceinline__ void vec_top_init(VecTop<DT, VW> &T) {
  T.best = Raw<DT, VW>{};
  T.bidx = -1;
  T.t1 = T.t2 = -__builtin_huge_valf();
}

// vm: the vector's maximum ignoring NaN; vidx its index in the row.
template <int DT, int VW>
__device__ __forceinline__ void vec_top_add(VecTop<DT, VW> &T,
                                            const Raw<DT, VW> &r, float vm,
                                            int vidx) {
  if (__builtin_expect(vm > T.t2, 0)) {
    if (vm > T.t1) {
      T.t2 = T.t1;
      T.t1 = vm;
      T.best = r;
      T.bidx = vidx;
    } else {
      T.t2 = vm;
    }
  }
}

template <int DT, int VW>
__device__ __forceinline__ void vec_top_store(const VecTop<DT, VW> &T,
                                              bool finite, uint4 *v, int *idx,
                                              float *t2) {
  __stcg(v, T.best.w);
  __stcg(idx, T.bidx);
  __stcg(t2, finite ? T.t2 : __builtin_huge_valf());
}

// The exact top-F of a row from the nrec thread records of a pass over it.
// Returns false, having written nothing, when they do not determine it;
// the caller then filters the whole row.  scratch holds kWarps * F keys,
// out F keys; *cta_th and *t2max are 0 on entry and on return.
// Block-wide.
template <int DT, int VW>
__device__ __forceinline__ bool cta_vec_topf(const uint4 *v, const int *idx,
                                             const float *t2, int nrec,
                                             uint32_t *cta_th, uint32_t *t2max,
                                             uint64_t *scratch, uint64_t *out,
                                             int F, int32_t *otok,
                                             float *olog,
                                             int32_t *dev_status) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  WarpFilter w;
  wf_init(w, F);
  bool inf = false;
  uint32_t tm = 0;
  // the next round's records are loaded while this round's are filtered
  uint4 nv = make_uint4(0u, 0u, 0u, 0u);
  int ni = -1;
  float nt = -__builtin_huge_valf();
  if ((int)threadIdx.x < nrec) {
    nv = __ldcg(v + threadIdx.x);
    ni = __ldcg(idx + threadIdx.x);
    nt = __ldcg(t2 + threadIdx.x);
  }
  for (int r0 = 0; r0 < nrec; r0 += kThreads) {  // block-uniform
    Raw<DT, VW> raw;
    raw.w = nv;
    const int vi = ni;
    const float t = nt;
    const int rn = r0 + kThreads + (int)threadIdx.x;
    if (rn < nrec) {
      nv = __ldcg(v + rn);
      ni = __ldcg(idx + rn);
      nt = __ldcg(t2 + rn);
    }
    if (!(t < __builtin_huge_valf())) inf = true;
    else if (t > -__builtin_huge_valf()) tm = max(tm, ord32(t));
    wf_sync(w, cta_th);
    wf_offer<DT, VW>(w, cta_th, raw, vi >= 0, vi * VW);
  }
  if (tm) atomicMax(t2max, tm);
  const bool anyinf = __syncthreads_or(inf) != 0;
  if (lane < F) scratch[warp * F + lane] = w.a;
  if (32 + lane < F) scratch[warp * F + 32 + lane] = w.b;
  __syncthreads();
  const int n = rank_keys(scratch, kWarps * F, F, out);
  const uint32_t T2 = *t2max;
  __syncthreads();
  if (threadIdx.x == 0) {
    *cta_th = 0;
    *t2max = 0;
  }
  const bool ok = !anyinf && n == F &&
                  (T2 == 0 || unord32(T2) < key_val(out[F - 1]));
  if (ok) fan_write(out, n, F, false, otok, olog, dev_status);
  __syncthreads();
  return ok;
}

}  // namespace sdv
