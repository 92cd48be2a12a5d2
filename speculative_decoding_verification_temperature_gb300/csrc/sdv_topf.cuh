// sdv_topf.cuh -- exact top-F selection of (logit, token id) pairs over a
// row slice, ordered by logit descending then id ascending (-0 == +0).
//
// Each warp keeps a sorted list of its best keys in registers (lane l holds
// entries l and 32 + l) and filters its elements against one CTA-wide
// threshold: the largest, over the warps, of each warp's F-th best value so
// far.  An element below it has F strictly better elements in that warp's
// list, which only ever improves, so it cannot be in the answer; elements at
// or above it (ties included, since another warp's equal value may carry a
// smaller token id) are inserted.  On the fast path a vector costs one
// compare of its maximum against the threshold and a warp vote.  The warps'
// lists are ranked together at the end.
//
// Before its first vector is filtered, a warp seeds its threshold with a
// value that at least F of its first elements reach (the F-th largest of
// the lanes' vector maxima, for F <= 32), so that the first round inserts
// about F keys instead of all of them.
#pragma once

#include "sdv_device.cuh"

namespace sdv {

// Order-preserving map of a non-NaN float to uint32 (-0 mapped like +0).
// Every non-NaN float maps above 0, which marks an empty key.
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

struct TopSmem {
  uint64_t flat[kWarps * SD_MAX_FANOUT];  // warps' lists / gathered lists
  uint64_t out[SD_MAX_FANOUT];            // result, descending
  uint32_t th;                            // ord32 of the CTA threshold, 0 = none
  int nan;
  // CTA-wide candidate buffer (cta_* below): flat[0..nbuf) holds keys
  // above thk
  uint64_t thk;
  int nbuf, tot;
};

// Per-thread view of its warp's filter.  All fields but nseen are
// warp-uniform.
struct WarpFilter {
  uint64_t a, b;  // list entries lane and 32 + lane (descending, 0 = empty)
  float th;       // filter threshold
  float nseen;    // NaN-propagating maximum of the lane's elements
  int F;
  bool two;       // list of 64 (F > 32)
  bool seeded;
};

__device__ __forceinline__ void wf_init(WarpFilter &w, int F) {
  w.a = 0;
  w.b = 0;
  w.th = -__builtin_huge_valf();
  w.nseen = -__builtin_huge_valf();
  w.F = F;
  w.two = F > 32;
  w.seeded = false;
}

__device__ __forceinline__ uint64_t shfl64(uint64_t v, int src) {
  const uint32_t lo = __shfl_sync(0xffffffffu, (uint32_t)v, src);
  const uint32_t hi = __shfl_sync(0xffffffffu, (uint32_t)(v >> 32), src);
  return ((uint64_t)hi << 32) | lo;
}
__device__ __forceinline__ uint64_t shfl_up64(uint64_t v) {
  const uint32_t lo = __shfl_up_sync(0xffffffffu, (uint32_t)v, 1);
  const uint32_t hi = __shfl_up_sync(0xffffffffu, (uint32_t)(v >> 32), 1);
  return ((uint64_t)hi << 32) | lo;
}

// Insert key x (the same in every lane) into the warp's sorted list; the
// last entry falls off.  Full warp.
__device__ __forceinline__ void wf_insert(WarpFilter &w, uint64_t x) {
  const int lane = threadIdx.x & 31;
  int p = __popc(__ballot_sync(0xffffffffu, w.a > x));
  if (w.two) {
    p += __popc(__ballot_sync(0xffffffffu, w.b > x));
    const uint64_t a31 = shfl64(w.a, 31);
    const uint64_t bu = shfl_up64(w.b);
    const int pb = 32 + lane;
    w.b = pb < p ? w.b : (pb == p ? x : (lane == 0 ? a31 : bu));
  }
  const uint64_t au = shfl_up64(w.a);
  w.a = lane < p ? w.a : (lane == p ? x : au);
}

// Raise the threshold to the F-th entry once the list holds F keys, and
// publish it to the CTA.  Full warp.
__device__ __forceinline__ void wf_raise(WarpFilter &w, uint32_t *cta_th) {
  const int f = w.F - 1;
  const uint64_t kf = f < 32 ? shfl64(w.a, f) : shfl64(w.b, f - 32);
  if (kf != 0) {
    const float v = key_val(kf);
    if (v > w.th) {
      w.th = v;
      if ((threadIdx.x & 31) == 0) atomicMax(cta_th, ord32(v));
    }
  }
}

// Pick up a higher threshold published by another warp (stale is fine: the
// published value only grows).
__device__ __forceinline__ void wf_sync(WarpFilter &w, const uint32_t *cta_th) {
  const uint32_t o = *(const volatile uint32_t *)cta_th;
  if (o != 0) w.th = fmaxf(w.th, unord32(o));
}

// Seed the threshold from each lane's largest value m1 and second largest
// m2 among its first elements (-inf for none; NaN never counts): the
// largest value s such that at least F of those elements reach it.  With
// F <= 32 the candidates are the m1 (F lanes reach s); with F > 32 the m2,
// counting both values of every lane.  Full warp.
__device__ __forceinline__ void wf_seed2(WarpFilter &w, float m1, float m2) {
  w.seeded = true;
  const float cand = w.two ? m2 : m1;
  int c = 0;
#pragma unroll 8
  for (int j = 0; j < 32; ++j) {
    const float a = __shfl_sync(0xffffffffu, m1, j);
    c += a >= cand;
    if (w.two) c += __shfl_sync(0xffffffffu, m2, j) >= cand;
  }
  float s = c >= w.F ? cand : -__builtin_huge_valf();
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    s = fmaxf(s, __shfl_xor_sync(0xffffffffu, s, o));
  w.th = fmaxf(w.th, s);
}

// Fold value z into a lane's two largest values (m1 >= m2; NaN skipped).
__device__ __forceinline__ void top2_add(float &m1, float &m2, float z) {
  const float lo = fminf(m1, z);  // fminf/fmaxf drop a NaN operand
  m1 = fmaxf(m1, z);
  m2 = fmaxf(m2, lo);
}

// The per-round seed: the lane's vector maxima.
template <int VW>
__device__ __forceinline__ void wf_seed_vec(WarpFilter &w, const float (&z)[VW]) {
  float m1 = -__builtin_huge_valf(), m2 = -__builtin_huge_valf();
#pragma unroll
  for (int e = 0; e < VW; ++e) top2_add(m1, m2, z[e]);
  wf_seed2(w, m1, m2);
}

// Offer VW values per lane (ok = false for idle lanes, whose values must be
// -inf); j0 is the token id of the first.  Full, converged warp.
template <int VW>
__device__ __forceinline__ void wf_offer_vals(WarpFilter &w, uint32_t *cta_th,
                                              const float (&z)[VW], bool ok,
                                              int j0) {
  const float vmax = vmax_nan_of<VW>(z);  // NaN: never >= th
  w.nseen = max_nan(w.nseen, vmax);
  if (__builtin_expect(!w.seeded, 0)) wf_seed_vec<VW>(w, z);
  if (__builtin_expect(__any_sync(0xffffffffu, vmax >= w.th), 0)) {
#pragma unroll
    for (int e = 0; e < VW; ++e) {
      const bool take = ok && z[e] >= w.th;
      unsigned m = __ballot_sync(0xffffffffu, take);
      if (m == 0) continue;
      const uint64_t key = make_key(ord32(z[e]), (uint32_t)(j0 + e));
      while (m) {
        const int src = __ffs(m) - 1;
        m &= m - 1;
        wf_insert(w, shfl64(key, src));
      }
      wf_raise(w, cta_th);
    }
  }
}

// Offer one vector of logits per lane.
template <int DT, int VW>
__device__ __forceinline__ void wf_offer(WarpFilter &w, uint32_t *cta_th,
                                         const Raw<DT, VW> &r, bool ok,
                                         int j0) {
  float z[VW];
#pragma unroll
  for (int e = 0; e < VW; ++e)
    z[e] = ok ? elt<DT, VW>(r, e) : -__builtin_huge_valf();
  wf_offer_vals<VW>(w, cta_th, z, ok, j0);
}

// Write the warp's best F keys to s.flat[warp * F ..].
__device__ __forceinline__ void wf_export(const WarpFilter &w, TopSmem &s) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t *dst = s.flat + warp * w.F;
  if (lane < w.F) dst[lane] = w.a;
  if (32 + lane < w.F) dst[32 + lane] = w.b;
}

// Rank the first C keys of s.flat (0 = empty, skipped) by counting and
// place the best F in s.out (descending).  Non-empty keys are unique.
// Returns min(F, non-empty keys); block-wide, every thread gets it.
__device__ __forceinline__ int rank_select(TopSmem &s, int C, int F) {
  int nz = 0;
  for (int i0 = 0; i0 < C; i0 += kThreads) {
    const int i = i0 + (int)threadIdx.x;
    const uint64_t me = i < C ? s.flat[i] : 0;
    if (me != 0) {
      int rank = 0;
      for (int j = 0; j < C; ++j) rank += s.flat[j] > me;
      if (rank < F) s.out[rank] = me;
    }
    nz += __syncthreads_count(me != 0);
  }
  __syncthreads();
  return nz < F ? nz : F;
}

// ------------------------------------------------------------------------
// CTA-wide candidate buffer, for large F.  The warp lists above keep each
// warp's own best F, so with F in the tens every warp inserts about F ln(n)
// keys one at a time.  Here the CTA keeps one buffer of candidates (the
// keys above thk, a lower bound on the CTA's F-th best) in s.flat; a chunk
// of elements costs one compare per element and an append per candidate,
// and the buffer is compacted to its best F (raising thk to the F-th) when
// a chunk's candidates would not fit.  Keys order as above.
constexpr int kCtaCap = kWarps * SD_MAX_FANOUT;
static_assert(SD_MAX_FANOUT + kThreads <= kCtaCap, "a round fits");

__device__ __forceinline__ void cta_reset(TopSmem &s) {
  if (threadIdx.x == 0) {
    s.th = 0;
    s.thk = 0;
    s.nbuf = 0;
    s.tot = 0;
  }
  __syncthreads();
}

// Sort a[0..n) (n <= kCtaCap) in descending order in place: a bitonic sort
// of the P = max(2, next power of two >= n) leading entries, a[n..P)
// padded with empty keys (which sort last); log2(P) (log2(P) + 1) / 2
// compare-exchange stages, threads < P / 2 taking one pair each.
// Block-wide.
__device__ __forceinline__ void cta_sort_desc(uint64_t *a, int n) {
  static_assert(kCtaCap <= 2 * kThreads, "one pair per thread per stage");
  int P = 2;
  while (P < n) P <<= 1;
  for (int i = n + (int)threadIdx.x; i < P; i += kThreads) a[i] = 0;
  __syncthreads();
  const int i = threadIdx.x;
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (i < P / 2) {
        const int lo = 2 * i - (i & (j - 1));  // pair (lo, lo + j)
        const int hi = lo + j;
        const uint64_t x = a[lo], y = a[hi];
        if ((x < y) == ((lo & k) == 0)) {  // descending where lo & k == 0
          a[lo] = y;
          a[hi] = x;
        }
      }
      __syncthreads();
    }
  }
}

// Merge nl lists of F keys each, every list descending with empty keys
// last, stored at a[l F ..]: a key's place in the union is its index in
// its own list plus, for every other list, the number of its keys above it
// (a binary search; non-empty keys are unique).  The best F go to out
// (descending); returns how many there are.  Block-wide.
__device__ __forceinline__ int cta_merge_lists(const uint64_t *a, int nl,
                                               int F, uint64_t *out) {
  int nz = 0;
  for (int i0 = 0; i0 < nl * F; i0 += kThreads) {
    const int idx = i0 + (int)threadIdx.x;
    const uint64_t me = idx < nl * F ? a[idx] : 0ull;
    if (me != 0) {
      const int l = idx / F;
      int r = idx - l * F;
      for (int o = 0; o < nl && r < F; ++o) {
        if (o == l) continue;
        const uint64_t *b = a + o * F;
        int lo = 0, hi = F;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (b[mid] > me) lo = mid + 1;
          else hi = mid;
        }
        r += lo;
      }
      if (r < F) out[r] = me;
    }
    nz += __syncthreads_count(me != 0);
  }
  __syncthreads();
  return nz < F ? nz : F;
}

// Compact s.flat[0..nbuf) (unique non-empty keys) to its best F, in
// descending order, and raise thk to the F-th.  Block-wide.
__device__ __forceinline__ void cta_compact(TopSmem &s, int F) {
  const int n = s.nbuf;
  cta_sort_desc(s.flat, n);
  if (threadIdx.x == 0) {
    const int m = n < F ? n : F;
    s.nbuf = m;
    if (m == F && s.flat[F - 1] > s.thk) s.thk = s.flat[F - 1];
  }
  __syncthreads();
}

// Seed thk from per-thread top-2 values (m1 >= m2; -inf for none) of the
// first elements: the F-th largest of these 2 kThreads samples has at least
// F elements at or above it, so keys of smaller value can be skipped.
// -inf samples may be placeholders and do not count.  Uses s.flat as
// scratch (one sort); leaves the buffer empty.  Block-wide.
__device__ __forceinline__ void cta_seed(TopSmem &s, float m1, float m2,
                                         int F) {
  const int t = threadIdx.x;
  // value keys made unique by their sample slot
  s.flat[2 * t] = m1 > -__builtin_huge_valf()
                      ? make_key(ord32(m1), (uint32_t)(2 * t)) : 0ull;
  s.flat[2 * t + 1] = m2 > -__builtin_huge_valf()
                          ? make_key(ord32(m2), (uint32_t)(2 * t + 1)) : 0ull;
  cta_sort_desc(s.flat, 2 * kThreads);
  if (t == 0 && s.flat[F - 1] != 0)  // admit values >= the F-th sample
    s.thk = ((s.flat[F - 1] >> 32) << 32) - 1ull;
  __syncthreads();
}

// Offer this thread's part of a chunk: vectors i = threadIdx.x, + kThreads,
// ... < cn of A, element ids (v0 + i) VW + e.  Returns whether a NaN was
// seen.  Block-wide.
template <int DT, int VW>
__device__ __forceinline__ bool cta_offer_chunk(TopSmem &s, const uint4 *A,
                                                int cn, int v0, int F) {
  const int t = threadIdx.x, lane = t & 31;
  const uint64_t thk = s.thk;
  // a key can beat thk only if its value reaches thk's (NaN never does)
  const float thv = thk ? unord32((uint32_t)(thk >> 32)) : -__builtin_huge_valf();
  int cnt = 0;
  bool nan = false;
  for (int i = t; i < cn; i += kThreads) {
    Raw<DT, VW> x;
    x.w = A[i];
#pragma unroll
    for (int e = 0; e < VW; ++e) {
      const float z = elt<DT, VW>(x, e);
      nan |= z != z;
      if (__builtin_expect(z >= thv, 0))
        cnt += make_key(ord32(z), (uint32_t)((v0 + i) * VW + e)) > thk;
    }
  }
  const int wsum = __reduce_add_sync(0xffffffffu, cnt);
  if (lane == 0 && wsum) atomicAdd(&s.tot, wsum);
  __syncthreads();
  const int tot = s.tot;
  if (tot == 0) return nan;  // block-uniform
  if (s.nbuf + tot > kCtaCap) cta_compact(s, F);
  const int nb = s.nbuf;
  __syncthreads();  // every thread has read nb before the appends below
  if (nb + tot <= kCtaCap) {  // append this chunk's candidates
    if (cnt) {
      int off = atomicAdd(&s.nbuf, cnt);
      for (int i = t; i < cn; i += kThreads) {
        Raw<DT, VW> x;
        x.w = A[i];
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          const float z = elt<DT, VW>(x, e);
          if (z >= thv) {
            const uint64_t k =
                make_key(ord32(z), (uint32_t)((v0 + i) * VW + e));
            if (k > thk) s.flat[off++] = k;
          }
        }
      }
    }
  } else {
    // more candidates than the buffer takes (ties, rising values): one
    // element per thread per round, compacting between rounds
    const int per = (cn + kThreads - 1) / kThreads;
    for (int u = 0; u < per; ++u) {
      const int i = t + u * kThreads;
      for (int e = 0; e < VW; ++e) {
        if (s.nbuf + kThreads > kCtaCap) cta_compact(s, F);
        const uint64_t th2 = s.thk;
        uint64_t k = 0;
        bool take = false;
        if (i < cn) {
          Raw<DT, VW> x;
          x.w = A[i];
          const float z = elt<DT, VW>(x, e);
          k = make_key(ord32(z), (uint32_t)((v0 + i) * VW + e));
          take = z == z && k > th2;
        }
        if (take) s.flat[atomicAdd(&s.nbuf, 1)] = k;
        __syncthreads();
      }
    }
  }
  __syncthreads();
  if (t == 0) s.tot = 0;
  return nan;
}

}  // namespace sdv
