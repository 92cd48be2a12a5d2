// sdv_topf.cuh -- exact top-F selection of (logit, token id) pairs over a
// row slice, ordered by logit descending then id ascending (-0 == +0).
//
// Streaming keeps a sorted top-kTopR list per thread (64-bit keys, one
// compare per element on the fast path).  The CTA then takes the F-th best
// of the per-thread maxima as a threshold, gathers the kept keys above it,
// ranks them by counting, and checks that no thread could have dropped a
// key that belongs in the result (a thread whose kTopR kept keys all reach
// the F-th result and that dropped something).  In that rare case the
// suspect threads rescan their own elements for a full top-F list and the
// selection is repeated over the union, which is exact.
#pragma once

#include "sdv_device.cuh"

namespace sdv {

constexpr int kTopR = 4;
constexpr int kTopCap = 2048;  // candidate list capacity (keys)

// Order-preserving map of a non-NaN float to uint32 (-0 mapped like +0).
__device__ __forceinline__ uint32_t ord32(float f) {
  const uint32_t u = __float_as_uint(f == 0.f ? 0.f : f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float unord32(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}
// Larger key = better: value first, then the smaller index.
__device__ __forceinline__ uint64_t make_key(uint32_t ord, uint32_t idx) {
  return ((uint64_t)ord << 32) | (uint32_t)(~idx);
}
__device__ __forceinline__ int key_idx(uint64_t k) { return (int)~(uint32_t)k; }
__device__ __forceinline__ float key_val(uint64_t k) {
  return unord32((uint32_t)(k >> 32));
}

struct TopR {
  uint64_t k[kTopR];  // descending; 0 = empty
  float thr;          // value of k[kTopR - 1] (-inf while not full)
  int nan;
  int dropped;
};

__device__ __forceinline__ void topr_init(TopR &t) {
#pragma unroll
  for (int r = 0; r < kTopR; ++r) t.k[r] = 0;
  t.thr = -__builtin_huge_valf();
  t.nan = 0;
  t.dropped = 0;
}

// Elements must be offered in increasing index order within a thread.
__device__ __forceinline__ void topr_add(TopR &t, float z, int j) {
  if (z != z) {
    t.nan = 1;
    return;
  }
  const uint32_t o = ord32(z);
  if (o <= (uint32_t)(t.k[kTopR - 1] >> 32)) {
    t.dropped |= (t.k[kTopR - 1] != 0);
    return;
  }
  t.dropped |= (t.k[kTopR - 1] != 0);
  uint64_t x = make_key(o, (uint32_t)j);
#pragma unroll
  for (int r = 0; r < kTopR; ++r) {
    const uint64_t hi = t.k[r] > x ? t.k[r] : x;
    const uint64_t lo = t.k[r] > x ? x : t.k[r];
    t.k[r] = hi;
    x = lo;
  }
  if (t.k[kTopR - 1] != 0) t.thr = key_val(t.k[kTopR - 1]);
}

// A vector: once the thread's list is full, one compare of the vector's
// maximum against the list's kTopR-th value on the fast path (an equal
// value comes later in index order, so it loses); NaN shows up in a packed
// sum of the vector (a vector holding both +inf and -inf also gives NaN
// there and is then checked element by element).
template <int DT, int VW>
__device__ __forceinline__ void topr_add_vec(TopR &t, const Raw<DT, VW> &r,
                                             int j0) {
  float z[VW];
#pragma unroll
  for (int e = 0; e < VW; ++e) z[e] = elt<DT, VW>(r, e);
  float chk;
  if constexpr (VW == 1) {
    chk = z[0];
  } else {
    float2 acc = make_float2(z[0], z[1]);
#pragma unroll
    for (int e = 2; e < VW; e += 2) acc = __fadd2_rn(acc, make_float2(z[e], z[e + 1]));
    chk = acc.x + acc.y;
  }
  const float vmax = vmax_of<VW>(z);
  const bool need = vmax > t.thr || t.k[kTopR - 1] == 0 || chk != chk;
  // vote so that the rare insertion is a real (warp-uniform) branch rather
  // than predicated work done for every element
  if (__builtin_expect(__any_sync(__activemask(), need), 0)) {
    if (need) {
#pragma unroll
      for (int e = 0; e < VW; ++e) topr_add(t, z[e], j0 + e);
    } else {
      t.dropped = 1;
    }
  } else {
    t.dropped = 1;
  }
}

struct TopSmem {
  uint64_t maxk[kThreads];
  uint64_t list[kTopCap];
  uint64_t out[SD_MAX_FANOUT];
  uint64_t theta0;
  int cnt;
  int nout;
};

// Rank the first C keys of `list` by counting and place the best F in out
// (descending).  Keys are unique.  Returns min(F, C).  Block-wide.
__device__ __forceinline__ int rank_select(TopSmem &s, int C, int F) {
  for (int i = threadIdx.x; i < C; i += kThreads) {
    const uint64_t me = s.list[i];
    int rank = 0;
    for (int j = 0; j < C; ++j) rank += s.list[j] > me;
    if (rank < F) s.out[rank] = me;
  }
  __syncthreads();
  return C < F ? C : F;
}

// Exact CTA-level top-F of the elements the threads offered to `mine`.
// `rescan(loc, F)` must rebuild this thread's own full top-F list (keys,
// descending, 0-padded) from its elements; it is called only by suspect
// threads.  Returns the number of keys in s.out; every thread gets it.
template <typename Rescan>
__device__ int cta_topf(const TopR &mine, int F, TopSmem &s, Rescan rescan) {
  const int tid = threadIdx.x;
  s.maxk[tid] = mine.k[0];
  if (tid == 0) {
    s.cnt = 0;
    s.theta0 = 1;  // fewer than F non-empty threads: take every key
  }
  __syncthreads();
  if (mine.k[0] != 0) {
    int rank = 0;
    for (int j = 0; j < kThreads; ++j) rank += s.maxk[j] > mine.k[0];
    if (rank == F - 1) s.theta0 = mine.k[0];
  }
  __syncthreads();
  const uint64_t th0 = s.theta0;
#pragma unroll
  for (int r = 0; r < kTopR; ++r)
    if (mine.k[r] != 0 && mine.k[r] >= th0) s.list[atomicAdd(&s.cnt, 1)] = mine.k[r];
  __syncthreads();
  int nout = rank_select(s, s.cnt, F);
  const uint64_t th = (nout == F) ? s.out[F - 1] : 1;
  const bool suspect =
      mine.dropped && (nout < F || mine.k[kTopR - 1] >= th);
  if (!__syncthreads_or(suspect)) return nout;

  // ---- rare: rebuild from full per-thread lists of the suspects ----
  __syncthreads();
  if (tid == 0) s.cnt = 0;
  __syncthreads();
  if (suspect) {
    uint64_t loc[SD_MAX_FANOUT];
    rescan(loc, F);
    for (int r = 0; r < F; ++r)
      if (loc[r] != 0 && loc[r] >= th) {
        const int pos = atomicAdd(&s.cnt, 1);
        if (pos < kTopCap) s.list[pos] = loc[r];
      }
  } else {
#pragma unroll
    for (int r = 0; r < kTopR; ++r)
      if (mine.k[r] != 0 && mine.k[r] >= th) {
        const int pos = atomicAdd(&s.cnt, 1);
        if (pos < kTopCap) s.list[pos] = mine.k[r];
      }
  }
  __syncthreads();
  const int C = s.cnt < kTopCap ? s.cnt : kTopCap;
  return rank_select(s, C, F);
}

// Insert a key into a descending local list of length F (suspect rescans).
__device__ __forceinline__ void local_insert(uint64_t *loc, int F, uint64_t x) {
  if (x <= loc[F - 1]) return;
  int r = F - 1;
  while (r > 0 && loc[r - 1] < x) {
    loc[r] = loc[r - 1];
    --r;
  }
  loc[r] = x;
}

}  // namespace sdv
