// sdv_filtered_any.cu -- linear verify with filtered sampling for any top_k
// (up to V) and any top_p ("01 · Draft-then-verify", section 4,
// standardised sampling: top-k and nucleus act on p and q first, and the
// ratio and the residual are formed from the adjusted distributions).
//
// The kept set of a row is a prefix of its tokens in (logit desc, id asc)
// order, so it is {j : K_j >= K*} for the composite key K_j = (ord(z_j) <<
// 32) | ~j and one threshold K*.  The kernel finds K* by a threshold select
// on the row itself, with no sort:
//
//  - One cluster verifies one sequence at a time (work counter).  At
//    position j every CTA brings its slices of the draft row j and the
//    target row j into shared memory with TMA bulk copies, where they stay
//    until the position is decided and, on a rejection, drawn from: each
//    row is read from HBM once.
//  - Row maximum m (cluster exchange), then a histogram of every finite
//    element by e = (m - z) log2(e) / T, the number of halvings of its
//    weight 2^-e below the maximum, in steps of 1/32 (1024 buckets, the last
//    one open-ended), holding counts and masses.  The CTAs' histograms are
//    summed range by range across the cluster (each CTA owns 1024 / CL
//    buckets), and every CTA finds the bucket where the criterion crosses:
//    the top_k-th element (counts), or the element at which the prefix mass
//    reaches top_p times the top-k mass (masses).
//  - The crossing bucket's elements are gathered into rank 0 (at most 256:
//    at the vocabularies of the pages a bucket holds tens), ranked exactly
//    by key, and the cut, its count and its mass follow from their prefix.
//    A larger bucket (ties of a constant row, or a deep top-k cut) is
//    refined first: histograms of (K_hi - K) >> shift over the candidates'
//    key interval, 1024 sub-buckets per level, until it fits.
//  - Top-k first (the k-th key and the top-k mass M_k), then the nucleus
//    against top_p M_k restricted to the top-k set; p~ = w / M over the kept
//    set with w = 2^(z k2 - m k2) and M the kept mass.
//  - The accept test r <= p~(x) / q~(x) from the two rows' thresholds and
//    masses; a rejection draws from norm(max(0, p~ - q~)) by inverse CDF
//    over the resident slices (segment masses, cluster prefix, one warp
//    scan), the bonus from p~_gamma.
#include "sdv_device.cuh"
#include "sdv_host.cuh"
#include "sdv_tma.cuh"
#include "sdv_topf.cuh"

namespace sdv {

constexpr int kFaNB = 1024;        // buckets per histogram level
constexpr float kFaRes = 32.f;     // level-1 buckets per halving of weight
constexpr int kFaG = 256;          // gathered candidates at most (one per thread)
constexpr int kFaMaxRange = kFaNB / 8;  // buckets a CTA owns (clusters >= 8)

struct FaParams {
  const void *target;  // [B, gamma+1, V]
  const void *draft;   // [B, gamma, V]
  const int32_t *tokens;
  const float *uniforms;
  int B, gamma, V;
  float k2;      // log2(e) / T
  int top_k;     // 1..V (V: no top-k cut)
  float top_p;   // (0, 1]
  int32_t *n_acc, *out_tokens;
  float *out_prob;
  int32_t *out_keep;  // [B, 2 gamma + 1] nullable: kept count per row read
  int32_t *dev_status;
  int *queue;
  int nclusters;
  int slice_vecs;  // capacity of one row's slice buffer (16-byte vectors)
  int seg_bytes;
};

// Selection state of one row (every CTA holds the same copy).
struct FaSel {
  int active;          // still searching
  int mass_mode;       // 0: count criterion, 1: mass criterion
  int level;           // 0: level-1 buckets; >= 1: key refinement
  int b1;              // level-1 bucket of the candidates (after level 1)
  int bmax;            // level 1, mass mode: last bucket allowed
  int shift;           // refinement digit shift
  uint64_t klo, khi;   // candidates' key interval (inclusive)
  uint32_t cnt_before; // elements ranked before the candidates
  double mass_before;  // their mass
  uint32_t tcount;     // count criterion: keep this many (>= 1)
  double tmass;        // mass criterion: prefix mass to reach
  uint32_t cand;       // candidates (cluster-wide)
  int gather;          // resolve by gathering at this step
  // result of the resolution
  uint64_t kcut;
  uint32_t count;
  double mass;
};

struct FaRow {
  float m;          // row maximum
  int bad;          // NaN / +inf, or no finite element
  uint32_t nfin;    // finite elements
  double total;     // their mass (weights relative to the maximum)
  uint64_t ks;      // final threshold (kept iff finite and K >= ks)
  double ms;        // kept mass
  float inv;        // 1 / ms (the draw multiplies: fp64 is slow)
  uint32_t ls;      // kept count
  uint64_t kk;      // top-k threshold
  double mk;        // top-k mass
  uint32_t lk;      // top-k count
  int bk;           // level-1 bucket of the top-k cut (kFaNB - 1 + 1: none)
};

struct FaSmem {
  // this CTA's range of buckets summed over the cluster: level 1 kept for
  // the nucleus search, refinement levels separately
  uint32_t rc1[2][kFaMaxRange];
  double rm1[2][kFaMaxRange];
  uint32_t rcx[2][kFaMaxRange];
  double rmx[2][kFaMaxRange];
  uint32_t tc1[2], tcx[2];  // range totals
  double tm1[2], tmx[2];
  // gathered candidates (rank 0's arrays are used)
  uint64_t gk[2][kFaG];
  float gw[2][kFaG];
  int gn[2][2];  // [gather parity][row]: appended candidates
  uint64_t res_k[2];
  uint32_t res_c[2];
  double res_m[2];
  // per-CTA partials of the row maximum (peers read), key range
  float pmax[2][2];  // [parity][row]
  int pbad[2][2];
  uint64_t pkmin[2], pkmax[2];
  FaSel sel[2];
  FaRow row[2];
  MS red[2][kWarps];
  float fred[kWarps][2];
  int ired[kWarps][2];
  uint64_t kred[kWarps][4];
  // position inputs
  int gx;
  float gr, gu, gzt, gzd;
  int kind, tok;
  float prob;
  int zero_mass;
  int next_seq[2];
  DrawSmem draw;
};

// Weight 2^(z k2 - m k2) of a logit and its level-1 bucket.
__device__ __forceinline__ float fa_weight(float z, float k2, float mk) {
  return ex2(fmaf(z, k2, -mk));
}
__device__ __forceinline__ int fa_bucket1(float z, float k2, float mk) {
  const float e = -fmaf(z, k2, -mk);
  const float s = e * kFaRes;
  return s >= (float)(kFaNB - 1) ? kFaNB - 1 : (s > 0.f ? (int)s : 0);
}

template <int DT, int VW>
__device__ __forceinline__ float fa_elt(const uint4 *buf, int i, int e) {
  Raw<DT, VW> r;
  r.w = buf[i];
  return elt<DT, VW>(r, e);
}

template <int DT, int VW>
__global__ void __launch_bounds__(kThreads, 2)
    filtered_any_kernel(const FaParams p) {
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ FaSmem sh;
  __shared__ uint64_t bar;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int CL = (int)cluster.num_blocks();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = p.V, gamma = p.gamma, G1 = gamma + 1, NS = 2 * gamma + 1;
  const float k2 = p.k2;
  const Slice sl = make_slice(V / VW, rank, CL);
  const int nv = sl.vend - sl.vbeg;
  const size_t rowb = (size_t)V * elt_bytes<DT>();
  // dynamic shared memory: the two rows' slices, segment masses, histograms
  uint4 *sbuf[2];
  sbuf[0] = reinterpret_cast<uint4 *>(dsm);
  sbuf[1] = sbuf[0] + p.slice_vecs;
  float *segmass = reinterpret_cast<float *>(sbuf[1] + p.slice_vecs);
  uint32_t *hc = reinterpret_cast<uint32_t *>(
      reinterpret_cast<unsigned char *>(segmass) + p.seg_bytes);  // [2][NB]
  float *hm = reinterpret_cast<float *>(hc + 2 * kFaNB);          // [2][NB]
  const int NR = kFaNB / CL;  // buckets this CTA owns
  const int r0 = rank * NR;
  uint32_t phase = 0;
  int par = 0, seqpar = 0;
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    sh.zero_mass = 0;
  }
  if (tid < 4) sh.gn[tid >> 1][tid & 1] = 0;
  int gpar = 0;  // parity of the next gather's counters
  __syncthreads();

  auto elem_key = [&](float z, int j) { return make_key(ord32(z), (uint32_t)j); };

  // -------- cluster-wide histogram steps ------------------------------------
  // Every thread: the histograms of the active rows (r in [rlo, rhi]) over
  // the candidates of the current level (fill(r, z, j, k) -> bucket or -1).
  auto hist_clear = [&]() {
    for (int i = tid; i < 2 * kFaNB; i += kThreads) {
      hc[i] = 0;
      hm[i] = 0.f;
    }
  };
  // Sum this CTA's range of buckets over the cluster (after a cluster
  // barrier that follows the fill) into rc/rm and the range totals.
  auto range_reduce = [&](int r, uint32_t *rc, double *rm, uint32_t &tcr,
                          double &tmr) {
    // GP consecutive threads per bucket, each reading every GP-th peer (the
    // remote loads are all in flight at once), then a shuffle sum in a
    // fixed order
    const int GP = kThreads / NR;  // 2 (clusters of 8) or 4 (16)
    {
      const int i = tid / GP, g = tid % GP;
      uint32_t c = 0;
      double m = 0.0;
#pragma unroll 4
      for (int q = g; q < CL; q += GP) {
        const uint32_t *phc = cluster.map_shared_rank(hc, q);
        const float *phm = cluster.map_shared_rank(hm, q);
        c += phc[r * kFaNB + r0 + i];
        m += (double)phm[r * kFaNB + r0 + i];
      }
      for (int o = 1; o < GP; o <<= 1) {
        c += __shfl_xor_sync(0xffffffffu, c, o);
        m += __shfl_xor_sync(0xffffffffu, m, o);
      }
      if (g == 0) {
        rc[i] = c;
        rm[i] = m;
      }
    }
    __syncthreads();
    if (warp == 0) {
      uint32_t c = 0;
      double m = 0.0;
      for (int i = lane; i < NR; i += 32) {
        c += rc[i];
        m += rm[i];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        c += __shfl_xor_sync(0xffffffffu, c, o);
        m += __shfl_xor_sync(0xffffffffu, m, o);
      }
      if (lane == 0) {
        tcr = c;
        tmr = m;
      }
    }
  };
  // One warp: find the bucket where the criterion of sel crosses, from the
  // range totals and ranges of every CTA (rc/rm/tc/tm of the given level
  // set).  Returns the bucket and its count / mass; adds the count / mass of
  // the buckets before it to sel.cnt_before / sel.mass_before.
  auto search = [&](FaSel &s, bool lvl1, int r, int bmax, int &bucket,
                    uint32_t &bc, double &bm) {
    // range totals of the CTAs, in rank order
    uint32_t c = 0;
    double m = 0.0;
    if (lane < CL) {
      const FaSmem *ps = cluster.map_shared_rank(&sh, lane);
      c = lvl1 ? ps->tc1[r] : ps->tcx[r];
      m = lvl1 ? ps->tm1[r] : ps->tmx[r];
    }
    uint32_t ci = c;
    double mi = m;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t uc = __shfl_up_sync(0xffffffffu, ci, o);
      const double um = __shfl_up_sync(0xffffffffu, mi, o);
      if (lane >= o) {
        ci += uc;
        mi += um;
      }
    }
    const uint32_t cbase = s.cnt_before;
    const double mbase = s.mass_before;
    // the first CTA range (up to bmax's range) whose inclusive prefix
    // crosses; rounding past the end: the last range with elements
    const int qmax = bmax / NR;
    bool hit;
    if (s.mass_mode) hit = lane < CL && lane <= qmax && mbase + mi >= s.tmass;
    else hit = lane < CL && lane <= qmax && cbase + ci >= s.tcount;
    unsigned hm_ = __ballot_sync(0xffffffffu, hit);
    int q;
    if (hm_) {
      q = __ffs(hm_) - 1;
    } else {
      const unsigned nz =
          __ballot_sync(0xffffffffu, lane < CL && lane <= qmax && c > 0);
      q = nz ? 31 - __clz(nz) : 0;
    }
    const uint32_t cb = __shfl_sync(0xffffffffu, ci - c, q);
    const double mb = __shfl_sync(0xffffffffu, mi - m, q);
    // inside CTA q's range
    const FaSmem *ps = cluster.map_shared_rank(&sh, q);
    const uint32_t *rcq = lvl1 ? ps->rc1[r] : ps->rcx[r];
    const double *rmq = lvl1 ? ps->rm1[r] : ps->rmx[r];
    uint32_t runc = cb;
    double runm = mb;
    int found = -1, lastnz = -1;
    uint32_t fc = 0, fcb = 0, lc = 0, lcb = 0;
    double fm = 0.0, fmb = 0.0, lm = 0.0, lmb = 0.0;
    const int lim = min(NR, bmax - q * NR + 1);
    for (int i0 = 0; i0 < lim && found < 0; i0 += 32) {
      const int i = i0 + lane;
      const uint32_t bc_ = i < lim ? rcq[i] : 0u;
      const double bm_ = i < lim ? rmq[i] : 0.0;
      uint32_t pc = bc_;
      double pm = bm_;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t uc = __shfl_up_sync(0xffffffffu, pc, o);
        const double um = __shfl_up_sync(0xffffffffu, pm, o);
        if (lane >= o) {
          pc += uc;
          pm += um;
        }
      }
      bool h;
      if (s.mass_mode) h = i < lim && bc_ > 0 && mbase + runm + pm >= s.tmass;
      else h = i < lim && cbase + runc + pc >= s.tcount;
      const unsigned hb = __ballot_sync(0xffffffffu, h);
      const unsigned nzb = __ballot_sync(0xffffffffu, i < lim && bc_ > 0);
      if (nzb) {
        const int L = 31 - __clz(nzb);
        lastnz = i0 + L;
        lc = __shfl_sync(0xffffffffu, bc_, L);
        lm = __shfl_sync(0xffffffffu, bm_, L);
        lcb = runc + __shfl_sync(0xffffffffu, pc - bc_, L);
        lmb = runm + __shfl_sync(0xffffffffu, pm - bm_, L);
      }
      if (hb) {
        const int L = __ffs(hb) - 1;
        found = i0 + L;
        fc = __shfl_sync(0xffffffffu, bc_, L);
        fm = __shfl_sync(0xffffffffu, bm_, L);
        fcb = runc + __shfl_sync(0xffffffffu, pc - bc_, L);
        fmb = runm + __shfl_sync(0xffffffffu, pm - bm_, L);
      }
      runc += __shfl_sync(0xffffffffu, pc, 31);
      runm += __shfl_sync(0xffffffffu, pm, 31);
    }
    if (found < 0) {  // rounding: the last bucket with elements
      found = lastnz < 0 ? 0 : lastnz;
      fc = lc;
      fm = lm;
      fcb = lcb;
      fmb = lmb;
    }
    bucket = q * NR + found;
    bc = fc;
    bm = fm;
    s.cnt_before = cbase + fcb;
    s.mass_before = mbase + fmb;
  };

  // Resolve the selections of the rows in [rlo, rhi]: level-1 search (the
  // level-1 ranges hold this position's histograms), then refinement levels
  // or a gather.  All threads of all CTAs call it.
  auto resolve = [&](int rlo, int rhi, const float *mk) {
    for (;;) {
      // ---- search at the current level (warp r for row r) ---------------
      if (warp >= rlo && warp <= rhi) {
        const int r = warp;
        FaSel s = sh.sel[r];
        if (s.active) {
          int bucket;
          uint32_t bc;
          double bm;
          const bool lvl1 = s.level == 0;
          search(s, lvl1, r, lvl1 ? s.bmax : kFaNB - 1, bucket, bc, bm);
          if (lvl1) {
            s.b1 = bucket;
            s.klo = 0;
            s.khi = ~0ull;
            if (s.mass_mode && bucket == sh.row[r].bk) {
              s.klo = sh.row[r].kk;  // inside the top-k set only
              bc = sh.row[r].lk - s.cnt_before;
            }
          } else {  // sub-bucket b holds keys in (khi - (b+1) 2^shift, khi - b 2^shift]
            const uint64_t hi = s.khi - ((uint64_t)bucket << s.shift);
            const uint64_t span = (s.shift >= 63) ? ~0ull
                                                  : ((1ull << s.shift) - 1);
            s.khi = hi;
            s.klo = (hi - s.klo > span) ? hi - span : s.klo;
          }
          s.cand = bc;
          s.gather = bc <= (uint32_t)kFaG || (s.level > 0 && s.shift == 0);
          ++s.level;
          if (lane == 0) sh.sel[r] = s;
        }
      }
      __syncthreads();
      bool any_refine = false, any_gather = false;
      for (int r = rlo; r <= rhi; ++r)
        if (sh.sel[r].active) {
          any_refine |= !sh.sel[r].gather;
          any_gather |= sh.sel[r].gather;
        }
      if (!any_refine && !any_gather) break;
      auto is_cand = [&](const FaSel &s, int r, float z, uint64_t k) {
        return z > -kInf && fa_bucket1(z, k2, mk[r]) == s.b1 && k >= s.klo &&
               k <= s.khi;
      };
      if (any_refine) {
        // key range of the refined rows' candidates, then one histogram
        // level over K - klo >> shift
        uint64_t kmin[2] = {~0ull, ~0ull}, kmax[2] = {0ull, 0ull};
        for (int r = rlo; r <= rhi; ++r) {
          const FaSel s = sh.sel[r];
          if (!s.active || s.gather) continue;
          for (int i = tid; i < nv; i += kThreads)
#pragma unroll
            for (int e = 0; e < VW; ++e) {
              const float z = fa_elt<DT, VW>(sbuf[r], i, e);
              const uint64_t k = elem_key(z, (sl.vbeg + i) * VW + e);
              if (is_cand(s, r, z, k)) {
                kmin[r] = min(kmin[r], k);
                kmax[r] = max(kmax[r], k);
              }
            }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            kmin[r] = min(kmin[r], (uint64_t)__shfl_xor_sync(
                                       0xffffffffu, (unsigned long long)kmin[r], o));
            kmax[r] = max(kmax[r], (uint64_t)__shfl_xor_sync(
                                       0xffffffffu, (unsigned long long)kmax[r], o));
          }
        if (lane == 0) {
          sh.kred[warp][0] = kmin[0];
          sh.kred[warp][1] = kmin[1];
          sh.kred[warp][2] = kmax[0];
          sh.kred[warp][3] = kmax[1];
        }
        __syncthreads();
        if (tid < 2) {
          uint64_t a = ~0ull, b = 0ull;
          for (int w = 0; w < kWarps; ++w) {
            a = min(a, sh.kred[w][tid]);
            b = max(b, sh.kred[w][2 + tid]);
          }
          sh.pkmin[tid] = a;
          sh.pkmax[tid] = b;
        }
        cluster.sync();
        if (warp < 2) {  // warp r merges row r's key range: lane q, CTA q
          const int r = warp;
          uint64_t a = ~0ull, b = 0ull;
          if (lane < CL) {
            const FaSmem *ps = cluster.map_shared_rank(&sh, lane);
            a = ps->pkmin[r];
            b = ps->pkmax[r];
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            a = min(a, (uint64_t)__shfl_xor_sync(0xffffffffu,
                                                 (unsigned long long)a, o));
            b = max(b, (uint64_t)__shfl_xor_sync(0xffffffffu,
                                                 (unsigned long long)b, o));
          }
          FaSel s = sh.sel[r];
          if (lane == 0 && r >= rlo && r <= rhi && s.active && !s.gather) {
            if (a > s.klo) s.klo = a;
            if (b < s.khi) s.khi = b;
            const uint64_t span = s.khi - s.klo;
            const int bits = span ? 64 - __clzll((long long)span) : 0;
            s.shift = bits > 10 ? bits - 10 : 0;
            sh.sel[r] = s;
          }
        }
        hist_clear();
        __syncthreads();
        for (int r = rlo; r <= rhi; ++r) {
          const FaSel s = sh.sel[r];
          if (!s.active || s.gather) continue;
          for (int i = tid; i < nv; i += kThreads)
#pragma unroll
            for (int e = 0; e < VW; ++e) {
              const float z = fa_elt<DT, VW>(sbuf[r], i, e);
              const uint64_t k = elem_key(z, (sl.vbeg + i) * VW + e);
              if (is_cand(s, r, z, k)) {
                const int b = (int)((s.khi - k) >> s.shift);  // 0: best
                atomicAdd(&hc[r * kFaNB + b], 1u);
                atomicAdd(&hm[r * kFaNB + b], fa_weight(z, k2, mk[r]));
              }
            }
        }
        cluster.sync();
        for (int r = rlo; r <= rhi; ++r) {
          const FaSel s = sh.sel[r];
          if (!s.active || s.gather) continue;
          range_reduce(r, sh.rcx[r], sh.rmx[r], sh.tcx[r], sh.tmx[r]);
          __syncthreads();
        }
        cluster.sync();
      }
      if (any_gather) {
        // every CTA appends the candidates of the gathering rows to rank 0
        // (counters of this parity were zeroed by rank 0 at the previous
        // gather, or at the start, before a cluster barrier)
        for (int r = rlo; r <= rhi; ++r) {
          const FaSel s = sh.sel[r];
          if (!s.active || !s.gather) continue;
          FaSmem *s0 = cluster.map_shared_rank(&sh, 0);
          for (int i = tid; i < nv; i += kThreads)
#pragma unroll
            for (int e = 0; e < VW; ++e) {
              const float z = fa_elt<DT, VW>(sbuf[r], i, e);
              const uint64_t k = elem_key(z, (sl.vbeg + i) * VW + e);
              if (is_cand(s, r, z, k)) {
                const int at = atomicAdd(&s0->gn[gpar][r], 1);
                if (at < kFaG) {
                  s0->gk[r][at] = k;
                  s0->gw[r][at] = fa_weight(z, k2, mk[r]);
                }
              }
            }
        }
        cluster.sync();
        if (rank == 0) {
          if (tid < 2) sh.gn[gpar ^ 1][tid] = 0;  // for the next gather
          for (int r = rlo; r <= rhi; ++r) {
            const FaSel s = sh.sel[r];
            if (!s.active || !s.gather) continue;
            const int n = min(sh.gn[gpar][r], kFaG);
            // rank by counting (keys are distinct), then scatter
            uint64_t k = 0;
            float w = 0.f;
            int pos = 0;
            if (tid < n) {
              k = sh.gk[r][tid];
              w = sh.gw[r][tid];
              for (int i = 0; i < n; ++i) pos += sh.gk[r][i] > k;
            }
            __syncthreads();
            if (tid < n) {
              sh.gk[r][pos] = k;
              sh.gw[r][pos] = w;
            }
            __syncthreads();
            if (warp == 0) {
              // inclusive prefix of the weights in key order; lane l holds
              // positions 8 l .. 8 l + 7
              double loc[kFaG / 32];
              double acc = 0.0;
#pragma unroll
              for (int e = 0; e < kFaG / 32; ++e) {
                const int i = lane * (kFaG / 32) + e;
                acc += i < n ? (double)sh.gw[r][i] : 0.0;
                loc[e] = acc;
              }
              double incl = acc;
#pragma unroll
              for (int o = 1; o < 32; o <<= 1) {
                const double u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
              }
              const double excl = incl - acc;
              int first = kFaG;
#pragma unroll
              for (int e = kFaG / 32 - 1; e >= 0; --e) {
                const int i = lane * (kFaG / 32) + e;
                bool h;
                if (s.mass_mode)
                  h = i < n && s.mass_before + excl + loc[e] >= s.tmass;
                else
                  h = i < n && s.cnt_before + (uint32_t)i + 1 >= s.tcount;
                if (h) first = i;
              }
#pragma unroll
              for (int o = 16; o > 0; o >>= 1)
                first = min(first, __shfl_xor_sync(0xffffffffu, first, o));
              if (first >= n) first = n - 1;  // rounding: keep them all
              if (first < 0) first = 0;       // (never: a bucket has one)
              const int src = first / (kFaG / 32), ei = first % (kFaG / 32);
              double mine = 0.0;
#pragma unroll
              for (int e = 0; e < kFaG / 32; ++e)
                if (e == ei) mine = excl + loc[e];
              const double pre = __shfl_sync(0xffffffffu, mine, src);
              if (lane == 0) {
                sh.res_k[r] = sh.gk[r][first];
                sh.res_c[r] = (uint32_t)(first + 1);
                sh.res_m[r] = pre;
              }
            }
            __syncthreads();
          }
        }
        cluster.sync();
        gpar ^= 1;
        if (tid < 2) {
          const int r = tid;
          FaSel s = sh.sel[r];
          if (r >= rlo && r <= rhi && s.active && s.gather) {
            const FaSmem *s0 = cluster.map_shared_rank(&sh, 0);
            s.kcut = s0->res_k[r];
            s.count = s.cnt_before + s0->res_c[r];
            s.mass = s.mass_before + s0->res_m[r];
            s.active = 0;
            sh.sel[r] = s;
          }
        }
        __syncthreads();
      }
    }
  };

  // -------- the sequences ----------------------------------------------
  int b = (int)(blockIdx.x / CL);
  while (b < p.B) {
    if (rank == 0 && tid == 0)
      sh.next_seq[seqpar] = p.nclusters + atomicAdd(p.queue, 1);
    int n = 0, kind = 0, bad_token = 0;
    for (int j = 0; j <= gamma; ++j) {
      const bool bonus = j == gamma;
      const int rlo = bonus ? 1 : 0;  // row 0: draft j, row 1: target j
      const char *rows[2] = {
          bonus ? nullptr
                : static_cast<const char *>(p.draft) +
                      ((size_t)b * gamma + j) * rowb,
          static_cast<const char *>(p.target) + ((size_t)b * G1 + j) * rowb};
      const uint32_t bytes = (uint32_t)nv * 16u;
      if (tid == 0) {
        fence_proxy_async();
        mbar_expect_tx(&bar, bytes * (bonus ? 1u : 2u));
        if (bytes) {
          if (!bonus)
            bulk_g2s(sbuf[0], rows[0] + (size_t)sl.vbeg * 16, bytes, &bar);
          bulk_g2s(sbuf[1], rows[1] + (size_t)sl.vbeg * 16, bytes, &bar);
        }
      }
      if (tid == 32) {  // the position's token, uniforms and gathers
        const int x = bonus ? 0 : p.tokens[(size_t)b * gamma + j];
        sh.gx = x;
        sh.gr = bonus ? 0.f : p.uniforms[(size_t)b * G1 + j];
        sh.gu = p.uniforms[(size_t)b * G1 + gamma];
        const bool ok = !bonus && x >= 0 && x < V;
        sh.gzt = ok ? load_logit<DT>(rows[1], x) : 0.f;
        sh.gzd = ok ? load_logit<DT>(rows[0], x) : 0.f;
      }
      mbar_wait(&bar, phase, p.dev_status);
      phase ^= 1;
      // ---- row maxima (NaN / +inf make the row unusable) ----------------
      {
        float mx[2] = {-kInf, -kInf};
        int bad[2] = {0, 0};
        for (int r = rlo; r < 2; ++r)
          for (int i = tid; i < nv; i += kThreads)
#pragma unroll
            for (int e = 0; e < VW; ++e) {
              const float z = fa_elt<DT, VW>(sbuf[r], i, e);
              bad[r] |= !(z < kInf) && !(z == -kInf);  // NaN or +inf
              mx[r] = fmaxf(mx[r], z);
            }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], o));
            bad[r] |= __shfl_xor_sync(0xffffffffu, bad[r], o);
          }
          if (lane == 0) {
            sh.fred[warp][r] = mx[r];
            sh.ired[warp][r] = bad[r];
          }
        }
        __syncthreads();
        if (tid < 2) {
          float a = -kInf;
          int bb = 0;
          for (int w = 0; w < kWarps; ++w) {
            a = fmaxf(a, sh.fred[w][tid]);
            bb |= sh.ired[w][tid];
          }
          sh.pmax[par][tid] = a;
          sh.pbad[par][tid] = bb;
        }
        cluster.sync();
        if (warp < 2) {  // warp r merges row r: lane q reads CTA q
          float a = -kInf;
          int bb = 0;
          if (lane < CL) {
            const FaSmem *ps = cluster.map_shared_rank(&sh, lane);
            a = ps->pmax[par][warp];
            bb = ps->pbad[par][warp];
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
            bb |= __shfl_xor_sync(0xffffffffu, bb, o);
          }
          if (lane == 0) {
            sh.row[warp].m = a;
            sh.row[warp].bad = bb || !(a > -kInf);
          }
        }
        par ^= 1;
        __syncthreads();
      }
      const bool unusable = sh.row[1].bad || (!bonus && sh.row[0].bad);
      if (unusable) {
        kind = 3;
        break;
      }
      const float mk[2] = {sh.row[0].m * k2, sh.row[1].m * k2};
      // ---- level-1 histograms of both rows ------------------------------
      hist_clear();
      __syncthreads();
      for (int r = rlo; r < 2; ++r)
        for (int i = tid; i < nv; i += kThreads)
#pragma unroll
          for (int e = 0; e < VW; ++e) {
            const float z = fa_elt<DT, VW>(sbuf[r], i, e);
            if (z > -kInf) {
              const int bk = fa_bucket1(z, k2, mk[r]);
              atomicAdd(&hc[r * kFaNB + bk], 1u);
              atomicAdd(&hm[r * kFaNB + bk], fa_weight(z, k2, mk[r]));
            }
          }
      cluster.sync();
      for (int r = rlo; r < 2; ++r) {
        range_reduce(r, sh.rc1[r], sh.rm1[r], sh.tc1[r], sh.tm1[r]);
        __syncthreads();
      }
      cluster.sync();
      // totals (warp r, lane q reads CTA q's range total, summed in a fixed
      // order), then the top-k selections
      if (warp < 2 && warp >= rlo) {
        const int r = warp;
        uint32_t c = 0;
        double m = 0.0;
        if (lane < CL) {
          const FaSmem *ps = cluster.map_shared_rank(&sh, lane);
          c = ps->tc1[r];
          m = ps->tm1[r];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          c += __shfl_xor_sync(0xffffffffu, c, o);
          m += __shfl_xor_sync(0xffffffffu, m, o);
        }
        if (lane == 0) {
          FaRow &R = sh.row[r];
          R.nfin = c;
          R.total = m;
          FaSel s = {};
          s.mass_mode = 0;
          s.bmax = kFaNB - 1;
          s.tcount = (uint32_t)p.top_k;
          s.active = (uint32_t)p.top_k < c;
          sh.sel[r] = s;
          if (!s.active) {  // no top-k cut: every finite token
            R.kk = 0;
            R.lk = c;
            R.mk = m;
            R.bk = kFaNB;  // no bucket holds the cut
          }
        }
      }
      __syncthreads();
      resolve(rlo, 1, mk);
      if (tid < 2 && tid >= rlo) {
        const int r = tid;
        FaRow &R = sh.row[r];
        const FaSel s = sh.sel[r];
        if ((uint32_t)p.top_k < R.nfin) {
          R.kk = s.kcut;
          R.lk = s.count;
          R.mk = s.mass;
          R.bk = s.b1;
        }
        // the nucleus over the top-k set
        FaSel t = {};
        t.mass_mode = 1;
        t.bmax = R.bk < kFaNB ? R.bk : kFaNB - 1;
        t.tmass = (double)p.top_p * R.mk;
        t.active = p.top_p < 1.f;
        sh.sel[r] = t;
        if (!t.active) {
          R.ks = R.kk;
          R.ls = R.lk;
          R.ms = R.mk;
        }
      }
      __syncthreads();
      resolve(rlo, 1, mk);
      if (tid < 2 && tid >= rlo && p.top_p < 1.f) {
        FaRow &R = sh.row[tid];
        const FaSel t = sh.sel[tid];
        R.ks = t.kcut > R.kk ? t.kcut : R.kk;
        R.ls = t.count;
        R.ms = t.mass;
      }
      __syncthreads();
      if (tid < 2 && tid >= rlo) sh.row[tid].inv = (float)(1.0 / sh.row[tid].ms);
      __syncthreads();
      if (rank == 0 && tid < 2 && tid >= rlo && p.out_keep)
        p.out_keep[(size_t)b * NS + (tid == 1 ? j : G1 + j)] =
            (int32_t)sh.row[tid].ls;
      // ---- the accept test ----------------------------------------------
      const FaRow Rt = sh.row[1], Rd = sh.row[0];
      const float k2m_t = mk[1], k2m_d = mk[0];
      auto ptil = [&](float z, int x, const FaRow &R, float mkr) {
        if (!(z > -kInf) || elem_key(z, x) < R.ks) return 0.0;
        return (double)fa_weight(z, k2, mkr) / R.ms;
      };
      if (!bonus) {
        if (tid == 0) {
          const int x = sh.gx;
          const bool bad = x < 0 || x >= V;
          int kd = 1;
          if (!bad) {
            const double pt = ptil(sh.gzt, x, Rt, k2m_t);
            const double qt = ptil(sh.gzd, x, Rd, k2m_d);
            const float rho = pt <= 0.0 ? 0.f
                              : (qt <= 0.0 ? kInf : (float)(pt / qt));
            kd = (double)sh.gr <= (double)rho && pt > 0.0 ? 0 : 1;
          }
          sh.kind = kd;
          bad_token |= bad;
        }
        __syncthreads();
        if (sh.kind == 0) {
          n = j + 1;
          continue;
        }
      }
      // ---- the draw: norm(max(0, p~ - q~)) on a rejection, p~ at the bonus
      {
        bool use_q = !bonus;
        const float u = sh.gu;
        DrawOut o;
        o.owner = -1;
        for (int attempt = 0; attempt < 2; ++attempt) {
          auto wgt = [&](int i, int e) {
            const int jj = (sl.vbeg + i) * VW + e;
            const float zt = fa_elt<DT, VW>(sbuf[1], i, e);
            float a = 0.f;
            if (zt > -kInf && elem_key(zt, jj) >= Rt.ks)
              a = __fmul_rn(fa_weight(zt, k2, k2m_t), Rt.inv);
            if (!use_q || a == 0.f) return a;
            const float zd = fa_elt<DT, VW>(sbuf[0], i, e);
            float q = 0.f;
            if (zd > -kInf && elem_key(zd, jj) >= Rd.ks)
              q = __fmul_rn(fa_weight(zd, k2, k2m_d), Rd.inv);
            return fmaxf(0.f, __fsub_rn(a, q));
          };
          cluster_total(cluster, sh.draw, segmass, sl, u, par, [&] {
            for (int s = warp; s < sl.nseg; s += kWarps) {
              const int i = s * 32 + lane;
              float acc = 0.f;
              if (i < nv)
#pragma unroll
                for (int e = 0; e < VW; ++e) acc += wgt(i, e);
              acc = warp_down_sum(acc);
              if (lane == 0) segmass[s] = acc;
            }
          });
          o.N = sh.draw.N;
          o.owner = sh.draw.owner;
          if (o.owner == rank) {
            if (tid == 0) {
              double tin = 0.0;
              sh.draw.seg = find_segment(segmass, sl.nseg, sh.draw.chunk_pre,
                                         sh.draw.tau, &tin);
              sh.draw.tau_seg = (float)tin;
            }
            __syncthreads();
            if (warp == 0) {
              const int i = sh.draw.seg * 32 + lane;
              float w[VW];
#pragma unroll
              for (int e = 0; e < VW; ++e) w[e] = i < nv ? wgt(i, e) : 0.f;
              float wt;
              const int t = warp_pick<VW>(w, sh.draw.tau_seg,
                                          (sl.vbeg + sh.draw.seg * 32) * VW,
                                          &wt);
              if (lane == 0) {
                sh.tok = t;
                sh.prob = (float)((double)wt / o.N);
              }
            }
          }
          if (o.owner >= 0) break;
          use_q = false;  // zero residual mass: draw from p~ instead
          sh.zero_mass = 1;
          __syncthreads();
        }
        __syncthreads();  // the owner's token and probability are visible
        kind = bonus ? 2 : 1;
        // the drawing CTA writes the outputs
        if (o.owner == rank && warp == 0) {
          for (int t = lane; t <= gamma; t += 32) {
            int v = -1;
            if (t < n) v = p.tokens[(size_t)b * gamma + t];
            else if (t == n) v = sh.tok;
            p.out_tokens[(size_t)b * G1 + t] = v;
          }
          if (lane == 0) {
            p.n_acc[b] = n;
            if (p.out_prob) p.out_prob[b] = sh.prob;
          }
        }
        __syncthreads();
      }
      break;
    }
    bad_token = __syncthreads_or(bad_token);
    if (rank == 0 && tid == 0) {
      int st = bad_token ? SD_DEV_BAD_TOKEN : 0;
      if (kind == 3) st |= SD_DEV_NONFINITE;
      else if (sh.zero_mass) st |= SD_DEV_ZERO_MASS;
      status_or(p.dev_status, st);
    }
    if (kind == 3 && rank == 0) {  // unusable row: outputs -1
      for (int t = tid; t <= gamma; t += kThreads)
        p.out_tokens[(size_t)b * G1 + t] = -1;
      if (tid == 0) {
        p.n_acc[b] = -1;
        if (p.out_prob) p.out_prob[b] = 0.f;
      }
    }
    if (rank == 0 && p.out_keep) {  // rows not read: -1
      for (int t = tid; t < NS; t += kThreads) {
        const bool tr = t <= gamma;
        const int jj = tr ? t : t - G1;
        const bool read = kind != 3 && (tr ? jj <= n : jj <= n && jj < gamma);
        if (!read) p.out_keep[(size_t)b * NS + t] = -1;
      }
    }
    __syncthreads();
    if (tid == 0) sh.zero_mass = 0;
    b = cluster.map_shared_rank(&sh, 0)->next_seq[seqpar];
    seqpar ^= 1;
    cluster.sync();  // every CTA has read next_seq before rank 0 rewrites it
  }
  cluster.sync();
}

}  // namespace sdv

namespace sdv {

using FaKernel = void (*)(const FaParams);

// Greedy filtered verify: the filters keep the argmax, so the kept count is
// 1 for every target row the greedy verify read (0..n) and -1 elsewhere.
__global__ void greedy_keep_kernel(const int32_t *n_acc, int B, int gamma,
                                   int32_t *out_keep) {
  const int NS = 2 * gamma + 1;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
       i < (long long)B * NS; i += (long long)gridDim.x * blockDim.x) {
    const int b = (int)(i / NS), t = (int)(i % NS);
    const int n = n_acc[b];
    out_keep[i] = (n >= 0 && t <= n) ? 1 : -1;
  }
}

sd_status greedy_keep(const int32_t *n_acc, int B, int gamma,
                      int32_t *out_keep, cudaStream_t s) {
  const long long total = (long long)B * (2 * gamma + 1);
  const long long blocks = (total + 255) / 256;
  const int grid = (int)(blocks < 1024 ? blocks : 1024);
  greedy_keep_kernel<<<grid, 256, 0, s>>>(n_acc, B, gamma, out_keep);
  SDV_CUDA(cudaGetLastError());
  return SD_OK;
}

// The general filtered verify (any top_k, any top_p).  Clusters of 8 or 16
// CTAs, the smallest whose CTAs hold both rows' slices in at most ~100 KB
// of shared memory (two CTAs per SM), else 16 with up to ~200 KB.
sd_status filtered_any_launch(const void *target, const void *draft,
                              sd_dtype dt, const int32_t *tokens,
                              const float *uniforms, int B, int gamma, int V,
                              float T, int top_k, float top_p, int32_t *n_acc,
                              int32_t *out_tokens, float *out_prob,
                              int32_t *out_keep, int32_t *dev_status,
                              void *ws, size_t ws_bytes, cudaStream_t s) {
  int sms = 0;
  sd_status st = check_device(&sms);
  if (st != SD_OK) return st;
  const int vw = dt == SD_F32 ? 4 : 8;
  const long long nvec = V / vw;
  FaKernel kern = dt == SD_F32 ? filtered_any_kernel<0, 4>
                               : filtered_any_kernel<1, 8>;
  auto smem_for = [&](int cl) {
    const long long per = (nvec + cl - 1) / cl;
    const size_t seg = ((size_t)((per + 31) / 32) * 4 + 127) / 128 * 128;
    return 2 * (size_t)per * 16 + seg + 2 * kFaNB * 8;
  };
  const int forced = tune(SD_TUNE_CLUSTER);
  int CL = (forced == 8 || forced == 16) ? forced
           : (smem_for(8) <= 100 * 1024 ? 8 : 16);
  const size_t smem = smem_for(CL);
  if (smem > 200 * 1024)
    return fail(SD_ERR_UNSUPPORTED,
                "V=%d: the filtered verify for top_k > %d or top_p < 1 "
                "holds a row pair in shared memory (%zu B per CTA needed)",
                V, SD_MAX_FANOUT, smem);
  int maxc = 0;
  st = max_active_clusters((const void *)kern, CL, smem, &maxc);
  if (st != SD_OK) return st;
  if (!ws || ws_bytes < 256)
    return fail(SD_ERR_INVALID_ARG, "workspace of >= 256 bytes required");
  const long long per = (nvec + CL - 1) / CL;
  FaParams prm;
  prm.target = target;
  prm.draft = draft;
  prm.tokens = tokens;
  prm.uniforms = uniforms;
  prm.B = B;
  prm.gamma = gamma;
  prm.V = V;
  prm.k2 = (float)(1.4426950408889634 / (double)T);
  prm.top_k = top_k < V ? top_k : V;
  prm.top_p = top_p;
  prm.n_acc = n_acc;
  prm.out_tokens = out_tokens;
  prm.out_prob = out_prob;
  prm.out_keep = out_keep;
  prm.dev_status = dev_status;
  prm.queue = static_cast<int *>(ws);
  prm.nclusters = B < maxc ? B : maxc;
  prm.slice_vecs = (int)per;
  prm.seg_bytes = (int)(((size_t)((per + 31) / 32) * 4 + 127) / 128 * 128);
  SDV_CUDA(cudaMemsetAsync(ws, 0, sizeof(int), s));
  void *args[] = {&prm};
  return launch_clusters((const void *)kern, prm.nclusters, CL, smem, s, args);
}

}  // namespace sdv
