// sdv_filtered.cu -- linear verify with filtered (top-k / nucleus) sampling
// ("01 · Draft-then-verify", section 4, standardised sampling: top-k and
// nucleus act on p and q first, and the ratio is formed from the adjusted
// distributions; Algorithm 1 otherwise unchanged).
//
// With top_k <= 64 everything the method needs about a row lives in its
// top_k (logit, id) keys: the filtered distribution is 2^((z - m) k2) over
// the kept keys (m the row maximum, k2 = log2(e)/T), the nucleus is a
// prefix of them, and the residual max(0, p~ - q~) is zero outside the
// target's kept tokens.  So each row is read from HBM once, and each CTA
// selects its slice's exact top-k: the ring pass keeps each thread's
// maximum, a bound follows from those maxima, and a second pass over the
// slice (from L2, just streamed) gathers and ranks the few elements at or
// above it.  The accept test, the correction and the bonus are computed by
// one warp on at most 64 keys per row.
//
// One thread-block cluster verifies one sequence at a time (work counter).
// Position j streams the CTAs' slices of the draft row j and the target row
// j back to back through the TMA ring (thread 0 issues the copies, the next
// position's only once position j was accepted); each CTA ranks its slice's
// candidates, the cluster exchanges the per-CTA lists through distributed
// shared memory, and every CTA ranks the CL lists of both rows into the
// rows' exact top-k.

// This kernel's ring: two stages of 16 KB.  Its CTAs then fit four to an SM
// (shared memory and 64 registers), and the more clusters in flight
// verify fewer sequences each one after another: on the large shape
// 149.8-153.5 us against 161.9-162.0 us with three stages and three CTAs
// per SM.  (No other translation unit sees this value.)
#define SDV_STAGES 2
#include "sdv_device.cuh"
#include "sdv_host.cuh"
#include "sdv_ring.cuh"
#include "sdv_tma.cuh"
#include "sdv_fanrow.cuh"
#include "sdv_topf.cuh"

namespace sdv {

struct FiltParams {
  const void *target;  // [B, gamma+1, V]
  const void *draft;   // [B, gamma, V]
  const int32_t *tokens;
  const float *uniforms;
  int B, gamma, V;
  float k2;     // log2(e) / T
  int top_k;    // 1..SD_MAX_FANOUT
  float top_p;  // (0, 1]
  int32_t *n_acc, *out_tokens;
  float *out_prob;
  int32_t *out_keep;  // [B, 2 gamma + 1] nullable: kept count per row read
  int32_t *dev_status;
  int *queue;
  int nclusters;
};

// Ring schedule (thread 0, shared memory).  Items: 0 draft row of position
// pj, 1 target row of position pj, 2 wait for decision pj, 3 the bonus row
// (target row gamma) when every position was accepted, 4 sequence done.
struct FSched {
  int pseq, pprev, pj, pkind;
  int dseq, decided, final, next;
};

struct FPState {
  const char *pa;
  int prem, issued;
};

struct FiltSmem {
  TopSmem top;
  uint64_t clist[2][2][SD_MAX_FANOUT];  // [parity][row]: this CTA's lists
  int cnan[2][2];                       // [parity][row]: a NaN in the slice
  uint64_t rk[2][SD_MAX_FANOUT];        // [row]: the rows' top-k (desc)
  int rnan[2];
  int next_seq[2];
  int gx;  // the position's draft token and uniforms (r, final u)
  float gr, gu;
  int kind;  // decision: 0 accept, 1 reject, 2 bonus drawn, 3 unusable
  int tok;
  float prob;
  int zero_mass;
  FSched sc;
  // the draw: kept target tokens sorted by id
  int dj[SD_MAX_FANOUT];
  float dw[SD_MAX_FANOUT];
};

template <int DT, int VW>
struct FFu {
  const FiltParams &p;
  const Slice &sl;
  Ring &rg;
  int nv;
  size_t rowb;

  __device__ const char *row(int kind, int b, int j) const {
    if (kind)
      return static_cast<const char *>(p.target) +
             ((size_t)b * (p.gamma + 1) + j) * rowb;
    return static_cast<const char *>(p.draft) + ((size_t)b * p.gamma + j) * rowb;
  }
  __device__ bool next_item(FSched &sc, FPState &ps) const {
    for (;;) {
      if (sc.pseq == -1) {
        if (sc.dseq != sc.pprev || sc.next < 0) return false;
        sc.pseq = sc.next;
      }
      if (sc.pseq >= p.B) return false;
      const bool cur = sc.pseq == sc.dseq;
      const int j = sc.pj;
      const char *ra = nullptr;
      if (sc.pkind == 0) {  // draft row j (after decision j-1)
        if (j >= p.gamma) {
          sc.pkind = 3;
          continue;
        }
        ra = row(0, sc.pseq, j);
        sc.pkind = 1;
      } else if (sc.pkind == 1) {
        ra = row(1, sc.pseq, j);
        sc.pkind = 2;
      } else if (sc.pkind == 2) {  // wait for decision j
        if (!(cur && sc.decided > j)) return false;
        if (sc.final) {
          sc.pkind = 4;
        } else {
          sc.pj = j + 1;
          sc.pkind = 0;
        }
        continue;
      } else if (sc.pkind == 3) {  // bonus: every position accepted
        ra = row(1, sc.pseq, p.gamma);
        sc.pkind = 4;
      } else {  // sequence done
        sc.pprev = sc.pseq;
        sc.pseq = -1;
        sc.pj = 0;
        sc.pkind = 0;
        continue;
      }
      if (nv > 0) {
        ps.pa = ra + (size_t)sl.vbeg * 16;
        ps.prem = nv;
        return true;
      }
    }
  }
  __device__ __forceinline__ void pump(FSched &sc, FPState &ps,
                                       int consumed) const {
    while (ps.issued < consumed + kStages) {
      if (ps.prem == 0 && !next_item(sc, ps)) return;
      const int cnt = min(kStageVecs, ps.prem);
      const uint32_t bytes = (uint32_t)cnt * 16u;
      const int s = ps.issued % kStages;
      fence_proxy_async();
      mbar_expect_tx(&rg.full[s], bytes);
      bulk_g2s(rg.buf + (size_t)s * kStageVecs, ps.pa, bytes, &rg.full[s]);
      ps.pa += bytes;
      ps.prem -= cnt;
      ++ps.issued;
    }
  }
};

template <class Fu, class F>
__device__ __forceinline__ void ft_consume(const Fu &fu, Ring &rg,
                                           FSched &sc, FPState &ps,
                                           int &consumed, uint32_t &phase,
                                           int32_t *dev_status, F &&f) {
  const int s = consumed % kStages;
  mbar_wait(&rg.full[s], (phase >> s) & 1u, dev_status);
  phase ^= 1u << s;
  f(rg.buf + (size_t)s * kStageVecs);
  __syncthreads();
  ++consumed;
  if (threadIdx.x == 0) fu.pump(sc, ps, consumed);
}

// The filtered distribution of a row from its top-k keys (descending, 0 =
// empty), for lane l: entries l and 32 + l.  e = 2^((v - m) k2) over the
// kept keys (the nucleus: a key stays while the mass before it, relative
// to the top-k mass, is below top_p), 0 elsewhere; returns Z = the kept
// mass (warp-uniform).  Warp 0 only.
struct FRow {
  float e0, e1;  // filtered (unnormalised) weights of entries lane, 32+lane
  int j0, j1;    // their token ids (-1: empty or dropped)
  float Z;
};

__device__ __forceinline__ float warp_incl_scan(float x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float up = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += up;
  }
  return x;
}

__device__ __forceinline__ FRow filtered_row(const uint64_t *keys, int k,
                                             float k2, float top_p) {
  const int lane = threadIdx.x & 31;
  FRow r;
  const uint64_t a = lane < k ? keys[lane] : 0ull;
  const uint64_t b = 32 + lane < k ? keys[32 + lane] : 0ull;
  const float m = key_val(keys[0]);
  const float mk = m * k2;
  float ea = a ? ex2(fmaf(key_val(a), k2, -mk)) : 0.f;
  float eb = b ? ex2(fmaf(key_val(b), k2, -mk)) : 0.f;
  // prefix masses in key order (entries 0..31 then 32..63)
  const float ca = warp_incl_scan(ea);
  const float ta = __shfl_sync(0xffffffffu, ca, 31);
  const float cb = warp_incl_scan(eb) + ta;
  const float tk = __shfl_sync(0xffffffffu, cb, 31);
  if (top_p < 1.f) {
    if (!((ca - ea) / tk < top_p)) ea = 0.f;
    if (!((cb - eb) / tk < top_p)) eb = 0.f;
  }
  r.e0 = ea;
  r.e1 = eb;
  r.j0 = ea > 0.f ? key_idx(a) : -1;
  r.j1 = eb > 0.f ? key_idx(b) : -1;
  float z = ea + eb;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  r.Z = z;
  return r;
}

// Kept tokens of a filtered row (warp-uniform).
__device__ __forceinline__ int fkept(const FRow &r) {
  return __popc(__ballot_sync(0xffffffffu, r.j0 >= 0)) +
         __popc(__ballot_sync(0xffffffffu, r.j1 >= 0));
}

// Filtered probability of token x in a row (warp-uniform; 0 if not kept).
__device__ __forceinline__ float fprob(const FRow &r, int x) {
  float v = (r.j0 == x ? r.e0 : 0.f) + (r.j1 == x ? r.e1 : 0.f);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v / r.Z;
}

// Inverse-CDF draw over the kept target tokens with weights w (per lane,
// entries lane and 32+lane; token ids j0/j1, -1 for none), in token-id
// order: the smallest id whose running sum exceeds u * N.  Writes the token
// and w_t / N into shared memory; returns N.  Warp 0 only.
__device__ __forceinline__ float fdraw(FiltSmem &sh, float w0, int j0,
                                       float w1, int j1, float u) {
  const int lane = threadIdx.x & 31;
  // rank each kept entry by id among the kept entries
  int r0 = 0, r1 = 0, cnt = 0;
  for (int src = 0; src < 32; ++src) {
    const int a = __shfl_sync(0xffffffffu, j0, src);
    const int b = __shfl_sync(0xffffffffu, j1, src);
    cnt += (a >= 0) + (b >= 0);
    r0 += (a >= 0 && a < j0) + (b >= 0 && b < j0);
    r1 += (a >= 0 && a < j1) + (b >= 0 && b < j1);
  }
  if (j0 >= 0) {
    sh.dj[r0] = j0;
    sh.dw[r0] = w0;
  }
  if (j1 >= 0) {
    sh.dj[r1] = j1;
    sh.dw[r1] = w1;
  }
  __syncwarp();
  const float x0 = lane < cnt ? sh.dw[lane] : 0.f;
  const float x1 = 32 + lane < cnt ? sh.dw[32 + lane] : 0.f;
  const float c0 = warp_incl_scan(x0);
  const float t0 = __shfl_sync(0xffffffffu, c0, 31);
  const float c1 = warp_incl_scan(x1) + t0;
  const float N = __shfl_sync(0xffffffffu, c1, 31);
  const float tau = u * N;
  unsigned h0 = __ballot_sync(0xffffffffu, lane < cnt && c0 > tau);
  unsigned h1 = __ballot_sync(0xffffffffu, 32 + lane < cnt && c1 > tau);
  int pos;
  if (h0) pos = __ffs(h0) - 1;
  else if (h1) pos = 32 + __ffs(h1) - 1;
  else {  // rounding: the last entry with mass
    const unsigned m0 = __ballot_sync(0xffffffffu, lane < cnt && x0 > 0.f);
    const unsigned m1 = __ballot_sync(0xffffffffu, 32 + lane < cnt && x1 > 0.f);
    pos = m1 ? 32 + 31 - __clz(m1) : (m0 ? 31 - __clz(m0) : 0);
  }
  if (lane == 0) {
    sh.tok = N > 0.f ? sh.dj[pos] : -1;
    sh.prob = N > 0.f ? sh.dw[pos] / N : 0.f;
  }
  __syncwarp();
  return N;
}

// The ring pass gives thread t the vectors at offsets t + kThreads m of its
// slice (a stage holds a multiple of kThreads vectors), which the re-read of
// a thread's part relies on.
static_assert(kStageVecs % kThreads == 0, "stage not a multiple of the CTA");

template <int DT, int VW>
__global__ void __launch_bounds__(kThreads, 4)
    filtered_verify_kernel(const FiltParams p) {
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ FiltSmem sh;
  __shared__ uint64_t bars[2 * kStages];
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int CL = (int)cluster.num_blocks();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = p.V, gamma = p.gamma, G1 = gamma + 1, K = p.top_k;
  const float k2 = p.k2;
  const Slice sl = make_slice(V / VW, rank, CL);
  Ring rg;
  rg.buf = reinterpret_cast<uint4 *>(dsm);
  rg.full = bars;
  rg.empty = bars + kStages;
  rg.dev_status = p.dev_status;
  const int nv = sl.vend - sl.vbeg;
  const int nch = (nv + kStageVecs - 1) / kStageVecs;
  const FFu<DT, VW> fu{p, sl, rg, nv, (size_t)V * elt_bytes<DT>()};

  int b = (int)(blockIdx.x / CL);
  if (tid == 0) {
    sh.top.th = 0;
    sh.sc = FSched{b, -1, 0, 0, b, 0, 0, -1};
  }
  ring_init(rg);  // (a block barrier)
  int par = 0, seqpar = 0, consumed = 0;
  uint32_t phase = 0;
  FPState ps{nullptr, 0, 0};
  auto consume = [&](auto &&f) {
    ft_consume(fu, rg, sh.sc, ps, consumed, phase, p.dev_status, f);
  };
  // One row through the ring into this CTA's list clist[par][r] (rowp:
  // the row in global memory).  During the ring pass each thread keeps the
  // vector holding its largest element (16 bytes in registers) and t2, the
  // largest maximum of its other vectors.  Each warp's ceil(K / kWarps)-th
  // largest lane maximum has that many of the warp's elements at or above
  // it, so the least of those over the warps, th, has at least K of the
  // slice's elements at or above it: the slice's best K are among the
  // elements >= th.  A thread with t2 < th holds all of its elements >= th
  // in its kept vector and appends them from registers.  The part of the
  // slice of any other thread is read again (from L2, just streamed) by
  // its whole warp, one vector per lane, and its elements >= th appended.
  // The gathered elements are ranked by counting.  When they overflow the
  // buffer (ties, rows of -inf), the candidate-buffer selection of
  // sdv_topf.cuh runs on the slice instead.
  auto select_row = [&](int r, const char *rowp) {
    VecTop<DT, VW> vt;
    vec_top_init(vt);
    bool nan = false;
    for (int c = 0; c < nch; ++c) {
      const int v0 = sl.vbeg + c * kStageVecs;
      const int cn = min(kStageVecs, nv - c * kStageVecs);
      consume([&](const uint4 *A) {
        for (int i = tid; i < cn; i += kThreads) {
          const Raw<DT, VW> x = sget<DT, VW>(A, i);
          float z[VW];
#pragma unroll
          for (int e = 0; e < VW; ++e) z[e] = elt<DT, VW>(x, e);
          const float vm = vmax_nan_of<VW>(z);
          nan |= vm != vm;
          vec_top_add(vt, x, vm, v0 + i);  // (a NaN maximum is not kept)
        }
      });
    }
    const float tmax = vt.t1;
    if (tid == 0) {
      sh.top.th = 0xffffffffu;
      sh.top.nbuf = 0;
    }
    const int anynan = __syncthreads_or(nan);
    {  // the warp's kw-th largest lane maximum; the least over the warps
      const int kw = (K + kWarps - 1) / kWarps;
      int cnt = 0;
      for (int l = 0; l < 32; ++l)
        cnt += __shfl_sync(0xffffffffu, tmax, l) >= tmax;
      float sv = cnt >= kw ? tmax : -__builtin_huge_valf();
      for (int o = 16; o; o >>= 1)
        sv = fmaxf(sv, __shfl_xor_sync(0xffffffffu, sv, o));
      if (lane == 0) atomicMin(&sh.top.th, ord32(sv));
    }
    __syncthreads();
    const float th = unord32(sh.top.th);
    const uint4 *src = reinterpret_cast<const uint4 *>(rowp) + sl.vbeg;
    if (!anynan) {
      auto append = [&](const Raw<DT, VW> &x, int vidx) {
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          const float z = elt<DT, VW>(x, e);
          if (z >= th) {
            const int slot = atomicAdd(&sh.top.nbuf, 1);
            if (slot < kCtaCap)
              sh.top.flat[slot] = make_key(ord32(z), (uint32_t)(vidx * VW + e));
          }
        }
      };
      const bool whole = !(vt.t2 < th);  // (also when th is -inf)
      if (!whole && vt.bidx >= 0 && vt.t1 >= th) append(vt.best, vt.bidx);
      // the parts of the threads with more than one vector reaching th
      for (unsigned m = __ballot_sync(0xffffffffu, whole); m; m &= m - 1) {
        const int owner = warp * 32 + __ffs(m) - 1;
        for (int i = owner + lane * kThreads; i < nv; i += 32 * kThreads) {
          Raw<DT, VW> x;
          x.w = __ldcg(src + i);
          append(x, sl.vbeg + i);
        }
      }
    }
    for (int i = tid; i < K; i += kThreads) sh.clist[par][r][i] = 0ull;
    __syncthreads();
    const int nc = sh.top.nbuf;
    if (nc <= kCtaCap) {  // rank the gathered elements (unique keys)
      for (int i = tid; i < nc; i += kThreads) {
        const uint64_t me = sh.top.flat[i];
        int rk = 0;
        for (int q = 0; q < nc; ++q) rk += sh.top.flat[q] > me;
        if (rk < K) sh.clist[par][r][rk] = me;
      }
    } else {  // too many: the candidate-buffer selection over the slice
      __syncthreads();  // every thread has read nc before the reset
      cta_reset(sh.top);
      for (int c = 0; c * kStageVecs < nv; ++c) {
        const int v0 = sl.vbeg + c * kStageVecs;
        const int cn = min(kStageVecs, nv - c * kStageVecs);
        const uint4 *A = src + c * kStageVecs;
        if (c == 0) {
          float m1 = -__builtin_huge_valf(), m2 = -__builtin_huge_valf();
          for (int i = tid; i < cn; i += kThreads) {
            Raw<DT, VW> x;
            x.w = __ldcg(A + i);
#pragma unroll
            for (int e = 0; e < VW; ++e) top2_add(m1, m2, elt<DT, VW>(x, e));
          }
          cta_seed(sh.top, m1, m2, K);
        }
        cta_offer_chunk<DT, VW>(sh.top, A, cn, v0, K);
      }
      cta_compact(sh.top, K);  // the slice's best K, descending
      const int nout = sh.top.nbuf;
      for (int i = tid; i < K; i += kThreads)
        sh.clist[par][r][i] = i < nout ? sh.top.flat[i] : 0ull;
    }
    if (tid == 0) {
      sh.cnan[par][r] = anynan;
      sh.top.th = 0;
    }
    __syncthreads();
  };
  // Exchange rows [r0, r0 + nr): every CTA ranks the CL lists of each row
  // into rk[r] (and rnan[r]).
  auto exchange = [&](int r0, int nr) {
    cluster.sync();
    for (int r = r0; r < r0 + nr; ++r) {
      if (tid == 0) sh.rnan[r] = 0;
      __syncthreads();
      for (int i = tid; i < CL * K; i += kThreads) {
        const FiltSmem *peer = cluster.map_shared_rank(&sh, i / K);
        sh.top.flat[i] = peer->clist[par][r][i % K];
        if (i % K == 0 && peer->cnan[par][r]) sh.rnan[r] = 1;
      }
      __syncthreads();
      const int n = cta_merge_lists(sh.top.flat, CL, K, sh.top.out);
      for (int i = tid; i < K; i += kThreads)
        sh.rk[r][i] = i < n ? sh.top.out[i] : 0ull;
      __syncthreads();
    }
    if (tid == 0 && sh.sc.next < 0)
      sh.sc.next = cluster.map_shared_rank(&sh, 0)->next_seq[seqpar];
    par ^= 1;
  };
  // A row is usable when it holds no NaN and its maximum is finite.
  auto row_ok = [&](int r) {
    const float m = sh.rk[r][0] ? key_val(sh.rk[r][0]) : -kInf;
    return !sh.rnan[r] && m > -kInf && m < kInf;
  };

  if (tid == 0) fu.pump(sh.sc, ps, consumed);
  while (b < p.B) {
    if (rank == 0 && tid == 0)
      sh.next_seq[seqpar] = p.nclusters + atomicAdd(p.queue, 1);
    int n = 0, bad_token = 0, kind = 0;
    for (int j = 0; j < gamma; ++j) {
      // the position's token and uniforms (warp 1; stored after the rows)
      int gx = 0;
      float gr = 0.f, gu = 0.f;
      if (tid == 32) {
        gx = p.tokens[(size_t)b * gamma + j];
        gr = p.uniforms[(size_t)b * G1 + j];
        gu = p.uniforms[(size_t)b * G1 + gamma];
      }
      select_row(0, fu.row(0, b, j));  // draft row j
      select_row(1, fu.row(1, b, j));  // target row j
      if (tid == 32) {
        sh.gx = gx;
        sh.gr = gr;
        sh.gu = gu;
      }
      exchange(0, 2);
      // the accept test of position j, on the last warp: warp 0 holds the
      // ring's producer (thread 0), whose own work would hold up the
      // warp-wide shuffles
      if (warp == kWarps - 1) {
        const int x = sh.gx;
        const bool bad = x < 0 || x >= V;
        int kd;
        if (!row_ok(0) || !row_ok(1)) {
          kd = 3;
        } else {
          const FRow fq = filtered_row(sh.rk[0], K, k2, p.top_p);
          const FRow fp = filtered_row(sh.rk[1], K, k2, p.top_p);
          const int kq = fkept(fq), kp = fkept(fp);
          if (p.out_keep && rank == 0 && lane == 0) {
            p.out_keep[(size_t)b * (2 * gamma + 1) + j] = kp;
            p.out_keep[(size_t)b * (2 * gamma + 1) + G1 + j] = kq;
          }
          const float px = bad ? 0.f : fprob(fp, x);
          const float qx = bad ? 0.f : fprob(fq, x);
          const float r = sh.gr;
          // p~(x) / q~(x); 0 when p~(x) == 0, +inf when only q~(x) == 0
          const bool acc = px > 0.f && (qx == 0.f || r <= px / qx);
          kd = acc ? 0 : 1;
          if (!acc) {  // the correction: norm(max(0, p~ - q~))
            float w0 = 0.f, w1 = 0.f;
            // q~ of each kept target token: search the draft's kept list
            float qa = 0.f, qb = 0.f;
            for (int src = 0; src < 32; ++src) {
              const int ja = __shfl_sync(0xffffffffu, fq.j0, src);
              const int jb = __shfl_sync(0xffffffffu, fq.j1, src);
              const float ea = __shfl_sync(0xffffffffu, fq.e0, src);
              const float eb = __shfl_sync(0xffffffffu, fq.e1, src);
              if (fp.j0 >= 0 && ja == fp.j0) qa += ea;
              if (fp.j0 >= 0 && jb == fp.j0) qa += eb;
              if (fp.j1 >= 0 && ja == fp.j1) qb += ea;
              if (fp.j1 >= 0 && jb == fp.j1) qb += eb;
            }
            if (fp.j0 >= 0)
              w0 = fmaxf(0.f, __fsub_rn(fp.e0 / fp.Z, qa / fq.Z));
            if (fp.j1 >= 0)
              w1 = fmaxf(0.f, __fsub_rn(fp.e1 / fp.Z, qb / fq.Z));
            const float u = sh.gu;
            float N = fdraw(sh, w0, w0 > 0.f ? fp.j0 : -1, w1,
                            w1 > 0.f ? fp.j1 : -1, u);
            int zm = 0;
            if (!(N > 0.f)) {  // zero residual mass: draw from p~ instead
              zm = 1;
              fdraw(sh, fp.e0, fp.j0, fp.e1, fp.j1, u);
            }
            if (lane == 0) sh.zero_mass = zm;
          }
        }
        if (lane == 0) sh.kind = kd;
        if (bad) bad_token = 1;
      }
      __syncthreads();
      kind = sh.kind;
      if (tid == 0) {  // the producer learns the decision
        FSched &sc = sh.sc;
        sc.decided = j + 1;
        if (kind) sc.final = 1;
        fu.pump(sc, ps, consumed);
      }
      if (kind) break;
      n = j + 1;
    }
    if (!kind) {  // every draft accepted: the bonus from p~_gamma
      select_row(1, fu.row(1, b, gamma));
      exchange(1, 1);
      if (warp == kWarps - 1) {
        int kd = 2;
        if (!row_ok(1)) {
          kd = 3;
        } else {
          const FRow fp = filtered_row(sh.rk[1], K, k2, p.top_p);
          const int kp = fkept(fp);
          if (p.out_keep && rank == 0 && lane == 0)
            p.out_keep[(size_t)b * (2 * gamma + 1) + gamma] = kp;
          fdraw(sh, fp.e0, fp.j0, fp.e1, fp.j1,
                p.uniforms[(size_t)b * G1 + gamma]);
          if (lane == 0) sh.zero_mass = 0;
        }
        if (lane == 0) sh.kind = kd;
      }
      __syncthreads();
      kind = sh.kind;
    }
    bad_token = __syncthreads_or(bad_token);
    if (rank == 0 && p.out_keep) {  // rows not read (or unusable): -1
      __syncthreads();
      const int NS = 2 * gamma + 1;
      for (int t = tid; t < NS; t += kThreads) {
        const bool tr = t <= gamma;
        const int jj = tr ? t : t - G1;
        const bool read = kind != 3 && (tr ? jj <= n : jj <= n && jj < gamma);
        if (!read) p.out_keep[(size_t)b * NS + t] = -1;
      }
    }
    if (rank == 0 && warp == 0) {  // outputs
      const bool unusable = kind == 3;
      for (int t = lane; t <= gamma; t += 32) {
        int v = -1;
        if (!unusable) {
          if (t < n) v = p.tokens[(size_t)b * gamma + t];
          else if (t == n) v = sh.tok;
        }
        p.out_tokens[(size_t)b * G1 + t] = v;
      }
      if (lane == 0) {
        p.n_acc[b] = unusable ? -1 : n;
        if (p.out_prob) p.out_prob[b] = unusable ? 0.f : sh.prob;
        status_or(p.dev_status, (bad_token ? SD_DEV_BAD_TOKEN : 0) |
                                    (unusable ? SD_DEV_NONFINITE : 0) |
                                    (!unusable && sh.zero_mass ? SD_DEV_ZERO_MASS : 0));
      }
    }
    __syncthreads();
    b = sh.sc.next;  // learnt at this sequence's first exchange
    seqpar ^= 1;
    __syncthreads();  // every thread has read it before thread 0 resets it
    if (tid == 0) {
      FSched &sc = sh.sc;
      sc.dseq = b;
      sc.decided = 0;
      sc.final = 0;
      sc.next = -1;
      fu.pump(sc, ps, consumed);
    }
    __syncthreads();
  }
  cluster.sync();  // no CTA leaves while a peer may still read its smem
}

using FiltKernel = void (*)(const FiltParams);

sd_status linear_launch(const void *target, const void *draft, sd_dtype dt,
                        long long d_seq_rows, const int32_t *tokens,
                        const float *uniforms, int B, int gamma, int V,
                        float T, int32_t *n_acc, int32_t *out_tokens,
                        float *out_prob, float *out_accept, float *out_resid,
                        int32_t *dev_status, void *ws, size_t ws_bytes,
                        cudaStream_t stream);

sd_status filtered_any_launch(const void *target, const void *draft,
                              sd_dtype dt, const int32_t *tokens,
                              const float *uniforms, int B, int gamma, int V,
                              float T, int top_k, float top_p, int32_t *n_acc,
                              int32_t *out_tokens, float *out_prob,
                              int32_t *out_keep, int32_t *dev_status,
                              void *ws, size_t ws_bytes, cudaStream_t s);
sd_status greedy_keep(const int32_t *n_acc, int B, int gamma,
                      int32_t *out_keep, cudaStream_t s);

}  // namespace sdv

extern "C" size_t sd_verify_linear_filtered_workspace(int B, int gamma,
                                                      int V, sd_dtype dt) {
  return sd_verify_linear_workspace(B, gamma, V, dt);
}

extern "C" sd_status sd_verify_linear_filtered(
    const void *target_logits, const void *draft_logits, sd_dtype dt,
    const int32_t *draft_tokens, const float *uniforms, int B, int gamma,
    int V, float T, int top_k, float top_p, int32_t *n_accepted,
    int32_t *out_tokens, float *out_prob, int32_t *out_keep,
    int32_t *dev_status, void *workspace, size_t ws_bytes, void *stream) {
  using namespace sdv;
  SDV_REQUIRE(dt == SD_F32 || dt == SD_BF16, "bad dtype %d", (int)dt);
  SDV_REQUIRE(B >= 0, "B < 0");
  SDV_REQUIRE(gamma >= 0 && gamma <= SD_MAX_GAMMA, "gamma=%d outside [0, %d]",
              gamma, SD_MAX_GAMMA);
  SDV_REQUIRE(V >= 1 && V <= SD_MAX_V, "V=%d outside [1, %d]", V, SD_MAX_V);
  SDV_REQUIRE(T >= 0.f && std::isfinite(T), "T must be finite and >= 0");
  SDV_REQUIRE(top_p > 0.f && top_p <= 1.f, "top_p outside (0, 1]");
  SDV_REQUIRE(top_k >= 1, "top_k=%d < 1", top_k);
  if (top_k > V) top_k = V;  // no top-k cut
  if (B == 0) return SD_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T == 0.f) {  // greedy: the filters keep the argmax
    sd_status g = linear_launch(target_logits, draft_logits, dt, gamma,
                                draft_tokens, uniforms, B, gamma, V, T,
                                n_accepted, out_tokens, out_prob, nullptr,
                                nullptr, dev_status, workspace, ws_bytes, s);
    if (g != SD_OK || !out_keep) return g;
    return greedy_keep(n_accepted, B, gamma, out_keep, s);
  }
  SDV_REQUIRE(target_logits && n_accepted && out_tokens && uniforms,
              "null pointer");
  SDV_REQUIRE(gamma == 0 || (draft_tokens && draft_logits),
              "draft tokens / logits are null");
  int sms = 0;
  sd_status st = check_device(&sms);
  if (st != SD_OK) return st;
  const int eb = dt == SD_F32 ? 4 : 2, vw = dt == SD_F32 ? 4 : 8;
  const bool vec = aligned16(target_logits) &&
                   (gamma == 0 || aligned16(draft_logits)) &&
                   ((size_t)V * eb) % 16 == 0;
  if (!vec)
    return fail(SD_ERR_UNSUPPORTED,
                "filtered verify needs 16-byte aligned rows (V * %d bytes)",
                eb);
  // top_k above the exact-list limit, or no top-k cut: the general kernel
  // (a threshold select on shared-memory resident rows)
  if (top_k > SD_MAX_FANOUT)
    return filtered_any_launch(target_logits, draft_logits, dt, draft_tokens,
                               uniforms, B, gamma, V, T, top_k, top_p,
                               n_accepted, out_tokens, out_prob, out_keep,
                               dev_status, workspace, ws_bytes, s);
  const long long nvec = V / vw;
  FiltKernel kern = dt == SD_F32 ? filtered_verify_kernel<0, 4>
                                 : filtered_verify_kernel<1, 8>;
  const size_t smem = kRingBytes;
  // clusters: the largest (a full stage per slice, CL * top_k keys gathered
  // in one rank) with at most ~2.5 sequences per resident cluster, else 1;
  // a cluster verifies its sequences one after another, and each row's
  // selection has a fixed cost, so a few sequences per cluster on larger
  // slices beat one sequence each on small ones (measured at B=256,
  // V=128256: clusters of 1, 2, 4 -> 463, 401, 374 us)
  int CL = 1, maxc = 0;
  const int forced = tune(SD_TUNE_CLUSTER);
  for (int c = 16; c >= 1; c /= 2) {
    if (forced && c != forced && c != 1) continue;
    if (c > 1 && nvec / c < kStageVecs && !forced) continue;
    if (c * top_k > kWarps * SD_MAX_FANOUT) continue;
    int mc = 0;
    st = max_active_clusters((const void *)kern, c, smem, &mc);
    if (st != SD_OK) return st;
    if (2LL * B <= 5LL * mc || c == 1 || forced) {
      CL = c;
      maxc = mc;
      break;
    }
  }
  if (maxc <= 0) return fail(SD_ERR_UNSUPPORTED, "no cluster fits");
  if (!workspace || ws_bytes < 256)
    return fail(SD_ERR_INVALID_ARG, "workspace of >= 256 bytes required");
  FiltParams prm;
  prm.target = target_logits;
  prm.draft = draft_logits;
  prm.tokens = draft_tokens;
  prm.uniforms = uniforms;
  prm.B = B;
  prm.gamma = gamma;
  prm.V = V;
  prm.k2 = (float)(1.4426950408889634 / (double)T);
  prm.top_k = top_k;
  prm.top_p = top_p;
  prm.n_acc = n_accepted;
  prm.out_tokens = out_tokens;
  prm.out_prob = out_prob;
  prm.out_keep = out_keep;
  prm.dev_status = dev_status;
  prm.queue = static_cast<int *>(workspace);
  prm.nclusters = B < maxc ? B : maxc;
  SDV_CUDA(cudaMemsetAsync(workspace, 0, sizeof(int), s));
  void *args[] = {&prm};
  return launch_clusters((const void *)kern, prm.nclusters, CL, smem, s, args);
}
