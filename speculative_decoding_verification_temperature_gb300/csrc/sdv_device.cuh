// sdv_device.cuh -- device building blocks shared by the verify kernels.
//
// Everything here is fp32 arithmetic on logits streamed from HBM: 16-byte
// read-only loads, bf16 widening, the online (max, sum) softmax state at
// temperature T, the greedy argmax state, warp / block reductions with a
// fixed combination order (so every CTA of a cluster that merges the same
// partials gets bit-identical results), and the three-level inverse-CDF
// draw (cluster slices -> 32-vector segments -> elements).
#pragma once

#include <cooperative_groups.h>
#include <cstdint>
#include <cuda_runtime.h>

#include "sd_verify.h"

namespace sdv {

namespace cg = cooperative_groups;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr float kInf = __builtin_huge_valf();

// ---------------------------------------------------------------- loads
// DT 0 = fp32, 1 = bf16.  VW = elements per load: 16 bytes (4 fp32 / 8
// bf16) on the vector path, 1 on the scalar path used when rows are not
// 16-byte aligned.
template <int DT, int VW> struct Raw;
template <> struct Raw<0, 4> { uint4 w; };
template <> struct Raw<1, 8> { uint4 w; };
template <> struct Raw<0, 1> { uint32_t w; };
template <> struct Raw<1, 1> { uint32_t w; };

template <int DT> __host__ __device__ constexpr int vec_width() { return DT == 0 ? 4 : 8; }
template <int DT> __host__ __device__ constexpr int elt_bytes() { return DT == 0 ? 4 : 2; }

__device__ __forceinline__ uint4 ld_nc_v4(const void *p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}
__device__ __forceinline__ uint32_t ld_nc_u32(const void *p) {
  uint32_t r;
  asm("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}
__device__ __forceinline__ uint32_t ld_nc_u16(const void *p) {
  unsigned short r;
  asm("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(r) : "l"(p));
  return (uint32_t)r;
}

// Load vector v (elements v*VW .. v*VW+VW-1) of a row.
template <int DT, int VW>
__device__ __forceinline__ Raw<DT, VW> load_vec(const void *row, int v) {
  Raw<DT, VW> r;
  if constexpr (VW > 1) {
    r.w = ld_nc_v4(static_cast<const char *>(row) + (size_t)v * 16);
  } else if constexpr (DT == 0) {
    r.w = ld_nc_u32(static_cast<const float *>(row) + v);
  } else {
    r.w = ld_nc_u16(static_cast<const uint16_t *>(row) + v);
  }
  return r;
}

// Element e of a loaded vector, widened to fp32 (bf16 widening is exact).
template <int DT, int VW>
__device__ __forceinline__ float elt(const Raw<DT, VW> &r, int e) {
  if constexpr (VW == 1) {
    return DT == 0 ? __uint_as_float(r.w) : __uint_as_float(r.w << 16);
  } else {
    const uint32_t words[4] = {r.w.x, r.w.y, r.w.z, r.w.w};
    if constexpr (DT == 0) {
      return __uint_as_float(words[e]);
    } else {
      const uint32_t u = words[e >> 1];
      return (e & 1) ? __uint_as_float(u & 0xffff0000u)
                     : __uint_as_float(u << 16);
    }
  }
}

// One logit at column j of a row (scalar, cached: used for gathers).
template <int DT>
__device__ __forceinline__ float load_logit(const void *row, int j) {
  if constexpr (DT == 0) return __ldg(static_cast<const float *>(row) + j);
  const unsigned short h = __ldg(static_cast<const unsigned short *>(row) + j);
  return __uint_as_float((uint32_t)h << 16);
}

// ------------------------------------------- programmatic dependent launch
// Wait until the grids this one depends on have completed and their writes
// are visible (a no-op when the kernel was launched without programmatic
// serialisation); let the next grid in the stream start launching.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" :::);
}

// ----------------------------------------------------------- fast exp2
// The SFU's approximate 2^x (ex2.approx, flush-to-zero): relative error a
// few ulp, far inside the 1e-5 decision margins the tests allow.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------- online softmax state
// Row statistics at temperature T with k2 = log2(e) / T:
//   m = max_j z_j,  s = sum_j 2^(z_j k2 - m k2)
// so that p_j = 2^(z_j k2 - m k2) / s.  The empty state holds m = kMEmpty
// (finite, below any usable logit) so the hot loop needs no test for
// "nothing seen yet": -inf entries add 2^-inf = 0.  NaN anywhere makes s
// NaN; +inf makes m infinite; a row of only -inf leaves m at kMEmpty and
// s = 0: all three are "invalid".
constexpr float kMEmpty = -3.0e38f;

struct MS {
  float m;
  float s;
};

__device__ __forceinline__ MS ms_empty() { return {kMEmpty, 0.f}; }

__device__ __forceinline__ MS ms_merge(MS a, MS b, float k2) {
  const float m = fmaxf(a.m, b.m);
  return {m, a.s * ex2((a.m - m) * k2) + b.s * ex2((b.m - m) * k2)};
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// NaN-propagating maxima (PTX max.NaN: NaN if any input is NaN).
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float max3_nan(float a, float b, float c) {
  float r;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Maximum of a vector that is NaN when any element is NaN.
template <int VW>
__device__ __forceinline__ float vmax_nan_of(const float (&z)[VW]) {
  if constexpr (VW == 1) {
    return z[0];
  } else if constexpr (VW == 4) {
    return max_nan(max3_nan(z[0], z[1], z[2]), z[3]);
  } else {
    return max3_nan(max3_nan(z[0], z[1], z[2]), max3_nan(z[3], z[4], z[5]),
                    max_nan(z[6], z[7]));
  }
}

template <int VW>
__device__ __forceinline__ float vmax_of(const float (&z)[VW]) {
  if constexpr (VW == 1) {
    return z[0];
  } else if constexpr (VW == 4) {
    return fmaxf(max3f(z[0], z[1], z[2]), z[3]);
  } else {
    return max3f(max3f(z[0], z[1], z[2]), max3f(z[3], z[4], z[5]),
                 fmaxf(z[6], z[7]));
  }
}

template <int DT, int VW>
__device__ __forceinline__ void ms_add_v(MS &st, const Raw<DT, VW> &r,
                                         float k2, float &vmax) {
  float z[VW];
#pragma unroll
  for (int e = 0; e < VW; ++e) z[e] = elt<DT, VW>(r, e);
  vmax = vmax_of<VW>(z);
  if (__builtin_expect(vmax > st.m, 0)) {  // rare once the large values are in
    st.s *= ex2((st.m - vmax) * k2);
    st.m = vmax;
  }
  // while nothing finite has been seen (m still the empty value, every
  // element so far -inf) the offset would overflow (-m k2 = +inf, and
  // -inf k2 + inf is NaN); 0 gives those elements their weight 0
  const float mk = st.m > kMEmpty ? -st.m * k2 : 0.f;
  if constexpr (VW == 1) {
    st.s += ex2(fmaf(z[0], k2, mk));
  } else {
    // packed fp32x2 arithmetic (two lanes per instruction)
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < VW; e += 2) {
      const float2 t = __ffma2_rn(make_float2(z[e], z[e + 1]),
                                  make_float2(k2, k2), make_float2(mk, mk));
      acc = __fadd2_rn(acc, make_float2(ex2(t.x), ex2(t.y)));
    }
    st.s += acc.x + acc.y;
  }
}

// The same, for callers that do not need the vector's maximum.
template <int DT, int VW>
__device__ __forceinline__ void ms_add(MS &st, const Raw<DT, VW> &r,
                                       float k2) {
  float vmax;
  ms_add_v<DT, VW>(st, r, k2, vmax);
}

// p(x)/q(x) of the draft token x from its target and draft logits zt, zd
// and the rows' merged states: 2^((zt - m_t) k2 - (zd - m_d) k2) s_d / s_t,
// with the same scaled exponents (fmaf(z, k2, -m k2)) that the draw's
// weights use.  Every verify kernel takes its accept test from here.
__device__ __forceinline__ float accept_ratio(float zt, float zd, MS mt,
                                             MS md, float k2) {
  const float e = fmaf(zt, k2, -mt.m * k2) - fmaf(zd, k2, -md.m * k2);
  return exp2f(e) * (md.s / mt.s);
}

__device__ __forceinline__ bool ms_valid(MS st) {
  return st.m > -1.0e38f && isfinite(st.m) && isfinite(st.s) && st.s > 0.f;
}

// --------------------------------------------------------- argmax state
// Greedy: largest logit, lowest index on ties; `bad` marks NaN / +inf.
struct AM {
  float v;
  int i;
  int bad;
};

__device__ __forceinline__ AM am_empty() { return {-kInf, 0x7fffffff, 0}; }

__device__ __forceinline__ AM am_merge(AM a, AM b) {
  AM r = (b.v > a.v || (b.v == a.v && b.i < a.i)) ? b : a;
  r.bad = a.bad | b.bad;
  return r;
}

template <int DT, int VW>
__device__ __forceinline__ void am_add(AM &st, const Raw<DT, VW> &r,
                                       int j0) {
#pragma unroll
  for (int e = 0; e < VW; ++e) {
    const float z = elt<DT, VW>(r, e);
    st.bad |= !(z < kInf);
    if (z > st.v) {
      st.v = z;
      st.i = j0 + e;
    }
  }
}

// ------------------------------------------------------ warp shuffles
__device__ __forceinline__ MS warp_down_ms(MS v, float k2) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    MS o{__shfl_down_sync(0xffffffffu, v.m, off),
         __shfl_down_sync(0xffffffffu, v.s, off)};
    v = ms_merge(v, o, k2);
  }
  return v;
}

__device__ __forceinline__ AM warp_down_am(AM v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    AM o{__shfl_down_sync(0xffffffffu, v.v, off),
         __shfl_down_sync(0xffffffffu, v.i, off),
         __shfl_down_sync(0xffffffffu, v.bad, off)};
    v = am_merge(v, o);
  }
  return v;
}

__device__ __forceinline__ float warp_down_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    v += __shfl_down_sync(0xffffffffu, v, off);
  return v;
}

// Block reduction of NR online states (result valid in thread 0).
template <int NR>
__device__ __forceinline__ void block_reduce_ms(MS (&v)[NR], float k2,
                                                MS (*scratch)[kWarps]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    v[r] = warp_down_ms(v[r], k2);
    if (lane == 0) scratch[r][warp] = v[r];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      MS a = scratch[r][0];
      for (int w = 1; w < kWarps; ++w) a = ms_merge(a, scratch[r][w], k2);
      v[r] = a;
    }
  }
}

__device__ __forceinline__ AM block_reduce_am(AM v, AM *scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_down_am(v);
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    AM a = scratch[0];
    for (int w = 1; w < kWarps; ++w) a = am_merge(a, scratch[w]);
    v = a;
  }
  return v;
}

// --------------------------------------------------------- slice layout
// A row of nvec vectors is cut into CL contiguous slices, one per CTA of
// the cluster; a slice is cut into segments of 32 consecutive vectors.
struct Slice {
  int vbeg, vend, nseg;
};

__device__ __forceinline__ Slice make_slice(int nvec, int rank, int CL) {
  Slice s;
  s.vbeg = (int)((long long)rank * nvec / CL);
  s.vend = (int)((long long)(rank + 1) * nvec / CL);
  s.nseg = (s.vend - s.vbeg + 31) >> 5;
  return s;
}

// ---------------------------------------- three-level inverse-CDF draw
// After every warp has written segmass[s] (fp32 sum of the weights of
// segment s), warp 0 forms 32 chunk sums (lane l: segments l*cs ..
// l*cs+cs-1, summed in order in double) and lane 0 their running total.
// chunk_pre[l] is the inclusive prefix; the slice total is chunk_pre[31].
__device__ __forceinline__ void slice_prefix(const float *segmass, int nseg,
                                             double *chunk_pre) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int cs = (nseg + 31) >> 5;
    double acc = 0.0;
    const int s0 = lane * cs, s1 = min(nseg, s0 + cs);
    for (int s = s0; s < s1; ++s) acc += (double)segmass[s];
    // inclusive prefix over the 32 chunk sums, in lane order
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double up = __shfl_up_sync(0xffffffffu, acc, o);
      if (lane >= o) acc += up;
    }
    chunk_pre[lane] = acc;
  }
}

// Find the segment holding the crossing C > tau inside this slice (tau
// relative to the slice start).  Returns the segment and writes the
// remaining target within it; falls back to the last segment with mass if
// rounding leaves no crossing.  Thread-0 only.
__device__ __forceinline__ int find_segment(const float *segmass, int nseg,
                                            const double *chunk_pre,
                                            double tau, double *tau_in_seg) {
  const int cs = (nseg + 31) >> 5;
  int l = 0;
  while (l < 31 && !(chunk_pre[l] > tau)) ++l;
  double before = l ? chunk_pre[l - 1] : 0.0;
  const int s0 = l * cs, s1 = min(nseg, s0 + cs);
  double acc = 0.0;
  for (int s = s0; s < s1; ++s) {
    const double nxt = acc + (double)segmass[s];
    if (nxt > tau - before) {
      *tau_in_seg = tau - before - acc;
      return s;
    }
    acc = nxt;
  }
  // no crossing (rounding at a chunk edge): last segment with mass in the
  // chunk, else in the slice
  for (int s = s1 - 1; s >= s0; --s)
    if (segmass[s] > 0.f) {
      *tau_in_seg = (double)segmass[s];
      return s;
    }
  for (int s = nseg - 1; s >= 0; --s)
    if (segmass[s] > 0.f) {
      *tau_in_seg = (double)segmass[s];
      return s;
    }
  *tau_in_seg = 0.0;
  return 0;
}

// Within one segment: given per-lane weights w[VW] (lane = vector index in
// the segment, ascending elements), return (in every lane) the element index
// of the first inclusive prefix > tau, or the last positive weight if none.
// out_w receives the chosen weight.
template <int VW>
__device__ __forceinline__ int warp_pick(const float (&w)[VW], float tau,
                                         int seg_first_elt, float *out_w) {
  const int lane = threadIdx.x & 31;
  float pre[VW];
  float run = 0.f;
#pragma unroll
  for (int e = 0; e < VW; ++e) {
    run += w[e];
    pre[e] = run;
  }
  // inclusive scan of lane totals
  float incl = run;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  const float excl = incl - run;
  int first = -1;
#pragma unroll
  for (int e = VW - 1; e >= 0; --e)
    if (excl + pre[e] > tau) first = e;
  const unsigned hit = __ballot_sync(0xffffffffu, first >= 0);
  int src_lane, src_e;
  if (hit) {
    src_lane = __ffs(hit) - 1;
    src_e = __shfl_sync(0xffffffffu, first, src_lane);
  } else {
    int lastpos = -1;
#pragma unroll
    for (int e = 0; e < VW; ++e)
      if (w[e] > 0.f) lastpos = e;
    const unsigned has = __ballot_sync(0xffffffffu, lastpos >= 0);
    src_lane = has ? 31 - __clz(has) : 0;
    src_e = __shfl_sync(0xffffffffu, has ? lastpos : 0, src_lane);
  }
  float mine = 0.f;
#pragma unroll
  for (int e = 0; e < VW; ++e)
    if (e == src_e) mine = w[e];
  *out_w = __shfl_sync(0xffffffffu, mine, src_lane);
  return seg_first_elt + src_lane * VW + src_e;
}

// ------------------------------------------------------- row accessors
// A row slice is read either straight from global memory (16-byte read-only
// loads, several in flight per thread) or from a copy a TMA bulk load put
// in shared memory.  Both give vector v (absolute index in the row).
template <int DT, int VW>
struct GRow {
  const char *p;
  static constexpr bool kSmem = false;
  __device__ __forceinline__ Raw<DT, VW> get(int v) const {
    return load_vec<DT, VW>(p, v);
  }
};

template <int DT, int VW>
struct SRow {
  const uint4 *p;  // shared copy of the slice, vector vbeg at p[0]
  int vbeg;
  static constexpr bool kSmem = true;
  __device__ __forceinline__ Raw<DT, VW> get(int v) const {
    Raw<DT, VW> r;
    r.w = p[v - vbeg];
    return r;
  }
};

// ------------------------------------------------------- streaming passes
constexpr int kU = 4;  // vectors per thread in flight per row (global)

// Accumulate the online softmax state of one or two rows over a slice.
template <int DT, int VW, class Row>
__device__ __forceinline__ void stats_pass(const Row &ra, const Row &rb,
                                           bool has_b, const Slice &sl,
                                           float k2, MS &a, MS &b) {
  if constexpr (Row::kSmem) {
    for (int v = sl.vbeg + (int)threadIdx.x; v < sl.vend; v += kThreads) {
      ms_add<DT, VW>(a, ra.get(v), k2);
      if (has_b) ms_add<DT, VW>(b, rb.get(v), k2);
    }
  } else {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int v0 = sl.vbeg + warp * 32 * kU + lane; v0 < sl.vend;
         v0 += kWarps * 32 * kU) {
      Raw<DT, VW> xa[kU], xb[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (v0 + u * 32 < sl.vend) {
          xa[u] = ra.get(v0 + u * 32);
          if (has_b) xb[u] = rb.get(v0 + u * 32);
        }
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (v0 + u * 32 < sl.vend) {
          ms_add<DT, VW>(a, xa[u], k2);
          if (has_b) ms_add<DT, VW>(b, xb[u], k2);
        }
    }
  }
}

// Accumulate the greedy argmax state of one row over a slice.
template <int DT, int VW, class Row>
__device__ __forceinline__ void argmax_pass(const Row &ra, const Slice &sl,
                                            AM &a) {
  if constexpr (Row::kSmem) {
    for (int v = sl.vbeg + (int)threadIdx.x; v < sl.vend; v += kThreads)
      am_add<DT, VW>(a, ra.get(v), v * VW);
  } else {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int v0 = sl.vbeg + warp * 32 * kU + lane; v0 < sl.vend;
         v0 += kWarps * 32 * kU) {
      Raw<DT, VW> xa[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (v0 + u * 32 < sl.vend) xa[u] = ra.get(v0 + u * 32);
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (v0 + u * 32 < sl.vend) am_add<DT, VW>(a, xa[u], (v0 + u * 32) * VW);
    }
  }
}

// Weights of a final draw: with a draft row,
//   w_j = max(0, p_j - c q_j) = max(0, 2^(zt k2 - mtk) ist - 2^(zd k2 - mdk) cq)
// (cq = c / s_q; c = 1 is the residual of section 2.1, c >= 1 the tree's
// repeated residual); without one, w_j = p_j = 2^(zt k2 - mtk) ist.
struct Weight {
  float k2, mtk, ist, mdk, cq;
};

template <int DT, int VW>
__device__ __forceinline__ void weights(const Raw<DT, VW> &a,
                                        const Raw<DT, VW> &b, bool has_q,
                                        const Weight &W, float (&w)[VW]) {
  // __fmul_rn keeps both products rounded before the subtraction (no FMA
  // contraction), so identical p and q rows give exactly zero residual.
#pragma unroll
  for (int e = 0; e < VW; ++e) {
    const float pt =
        __fmul_rn(ex2(fmaf(elt<DT, VW>(a, e), W.k2, -W.mtk)), W.ist);
    if (has_q) {
      const float qd =
          __fmul_rn(ex2(fmaf(elt<DT, VW>(b, e), W.k2, -W.mdk)), W.cq);
      w[e] = fmaxf(0.f, __fsub_rn(pt, qd));
    } else {
      w[e] = pt;
    }
  }
}

// Per-segment masses of the weights over this CTA's slice (segment s =
// vectors vbeg + 32 s .. vbeg + 32 s + 31; one warp per segment).
template <int DT, int VW, class Row>
__device__ __forceinline__ void mass_pass(const Row &ra, const Row &rb,
                                          bool has_q, const Weight &W,
                                          const Slice &sl, float *segmass) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int UU = Row::kSmem ? 1 : kU;
  for (int s0 = warp; s0 < sl.nseg; s0 += kWarps * UU) {
    Raw<DT, VW> xa[UU], xb[UU];
#pragma unroll
    for (int u = 0; u < UU; ++u) {
      const int v = sl.vbeg + (s0 + u * kWarps) * 32 + lane;
      if (s0 + u * kWarps < sl.nseg && v < sl.vend) {
        xa[u] = ra.get(v);
        if (has_q) xb[u] = rb.get(v);
      }
    }
#pragma unroll
    for (int u = 0; u < UU; ++u) {
      const int s = s0 + u * kWarps;
      if (s < sl.nseg) {  // warp-uniform
        const int v = sl.vbeg + s * 32 + lane;
        float acc = 0.f;
        if (v < sl.vend) {
          float w[VW];
          weights<DT, VW>(xa[u], xb[u], has_q, W, w);
#pragma unroll
          for (int e = 0; e < VW; ++e) acc += w[e];
        }
        acc = warp_down_sum(acc);
        if (lane == 0) segmass[s] = acc;
      }
    }
  }
}

// Shared state of a cluster-wide inverse-CDF draw (one per CTA).
constexpr int kMaxCL = 16;  // CTAs per cluster

struct DrawSmem {
  double slice[2];  // [parity] this CTA's slice mass (peers read)
  double chunk_pre[32];
  double N;      // total mass (all CTAs agree)
  double tau;    // u * N minus the mass of the slices before the owner
  int owner;     // CTA holding the crossing (-1: zero mass)
  int seg;       // owner: segment of the crossing
  float tau_seg; // owner: target left inside that segment
};

struct DrawOut {
  double N;
  int owner;
  int t;     // warp 0 of the owner CTA: drawn token
  float wt;  // its weight (probability wt / N)
};

// Cluster-wide total of the weights over the row(s): `fill()` makes every
// CTA write its per-segment masses, then the slice totals are exchanged
// (one cluster barrier) and warp 0 of every CTA forms their running sums in
// rank order (all CTAs do the same arithmetic, so all agree).  With u in
// (0, 1) it also finds the CTA whose slice holds the crossing C > u N and
// the target left in it.  Every thread of every CTA must call it.
template <class Fill>
__device__ double cluster_total(cg::cluster_group &cluster, DrawSmem &ds,
                                float *segmass, const Slice &sl, float u,
                                int &par, Fill &&fill) {
  const int tid = threadIdx.x;
  const int CL = (int)cluster.num_blocks();
  fill();
  __syncthreads();
  slice_prefix(segmass, sl.nseg, ds.chunk_pre);
  __syncthreads();
  if (tid == 0) ds.slice[par] = sl.nseg ? ds.chunk_pre[31] : 0.0;
  cluster.sync();
  if (tid < 32) {
    // lane r reads slice r; running sums in rank order
    const int lane = tid;
    const double sr =
        lane < CL ? cluster.map_shared_rank(&ds, lane)->slice[par] : 0.0;
    double pre = sr;  // inclusive prefix of the slice masses, rank order
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double up = __shfl_up_sync(0xffffffffu, pre, o);
      if (lane >= o) pre += up;
    }
    const double up1 = __shfl_up_sync(0xffffffffu, pre, 1);
    const double before = lane ? up1 : 0.0;
    const double tot = __shfl_sync(0xffffffffu, pre, 31);
    const double tau = (double)u * tot;
    unsigned hit = __ballot_sync(0xffffffffu, lane < CL && pre > tau);
    if (!hit && tot > 0.0)  // rounding: last slice with mass
      hit = 1u << (31 - __clz(__ballot_sync(0xffffffffu, lane < CL && sr > 0.0)));
    const int own = hit ? __ffs(hit) - 1 : -1;
    const double bef = __shfl_sync(0xffffffffu, before, own < 0 ? 0 : own);
    if (lane == 0) {
      ds.N = tot;
      ds.owner = tot > 0.0 ? own : -1;
      ds.tau = tau - bef;
    }
  }
  __syncthreads();
  par ^= 1;
  return ds.N;
}

template <int DT, int VW, class Row>
__device__ double cluster_mass(cg::cluster_group &cluster, DrawSmem &ds,
                               float *segmass, const Row &ra, const Row &rb,
                               bool has_q, const Weight &W, const Slice &sl,
                               float u, int &par) {
  return cluster_total(cluster, ds, segmass, sl, u, par, [&] {
    mass_pass<DT, VW>(ra, rb, has_q, W, sl, segmass);
  });
}

// After cluster_total: the owner CTA finds the segment of the crossing and
// one warp scans it (reading the vectors through `ra` / `rb`).
template <int DT, int VW, class Row>
__device__ DrawOut draw_pick(cg::cluster_group &cluster, DrawSmem &ds,
                             const float *segmass, const Row &ra,
                             const Row &rb, bool has_q, const Weight &W,
                             const Slice &sl) {
  const int tid = threadIdx.x;
  const int rank = (int)cluster.block_rank();
  DrawOut out;
  out.N = ds.N;
  out.owner = ds.owner;
  out.t = -1;
  out.wt = 0.f;
  if (out.owner == rank) {
    if (tid == 0) {
      double tin = 0.0;
      ds.seg = find_segment(segmass, sl.nseg, ds.chunk_pre, ds.tau, &tin);
      ds.tau_seg = (float)tin;
    }
    __syncthreads();
    if (tid < 32) {
      const int s = ds.seg;
      const int v = sl.vbeg + s * 32 + tid;
      float w[VW];
      if (v < sl.vend) {
        Raw<DT, VW> a = ra.get(v), b;
        if (has_q) b = rb.get(v);
        weights<DT, VW>(a, b, has_q, W, w);
      } else {
#pragma unroll
        for (int e = 0; e < VW; ++e) w[e] = 0.f;
      }
      out.t = warp_pick<VW>(w, ds.tau_seg, (sl.vbeg + s * 32) * VW, &out.wt);
    }
  }
  return out;
}

// Draw one token from the weights W over the row(s) by inverse CDF with
// uniform u: the smallest j with C_j > u * N.  Every thread of every CTA of
// the cluster must call it (it holds one cluster barrier); `par` is the
// caller's parity of the double-buffered slot.
template <int DT, int VW, class Row>
__device__ DrawOut cluster_draw(cg::cluster_group &cluster, DrawSmem &ds,
                                float *segmass, const Row &ra, const Row &rb,
                                bool has_q, const Weight &W, const Slice &sl,
                                float u, int &par) {
  cluster_mass<DT, VW>(cluster, ds, segmass, ra, rb, has_q, W, sl, u, par);
  return draw_pick<DT, VW>(cluster, ds, segmass, ra, rb, has_q, W, sl);
}

// Debug output: the normalised weights w_j / N over this CTA's slice.
template <int DT, int VW, class Row>
__device__ __forceinline__ void write_resid(float *res, const Row &ra,
                                            const Row &rb, bool has_q,
                                            const Weight &W, const Slice &sl,
                                            double N) {
  const float invN = (float)(1.0 / N);
  for (int v = sl.vbeg + threadIdx.x; v < sl.vend; v += kThreads) {
    Raw<DT, VW> a = ra.get(v), b;
    if (has_q) b = rb.get(v);
    float w[VW];
    weights<DT, VW>(a, b, has_q, W, w);
#pragma unroll
    for (int e = 0; e < VW; ++e) res[(size_t)v * VW + e] = w[e] * invN;
  }
}

// GPU-scope accesses to flags and counters that other CTAs write while this
// kernel runs (a plain load could be served from a stale L1 line)
__device__ __forceinline__ int ld_acquire_gpu(const int *a) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(a)
               : "memory");
  return v;
}
__device__ __forceinline__ int ld_relaxed_gpu(const int *a) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(a)
               : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(int *a, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(a), "r"(v)
               : "memory");
}
__device__ __forceinline__ void st_relaxed_gpu(int *a, int v) {
  asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(a), "r"(v)
               : "memory");
}

__device__ __forceinline__ void status_or(int32_t *dev_status, int bits) {
  if (dev_status && bits) atomicOr(dev_status, bits);
}

}  // namespace sdv
