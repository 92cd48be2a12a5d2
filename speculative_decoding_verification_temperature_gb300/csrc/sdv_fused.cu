// sdv_fused.cu -- linear verify ("01 · Draft-then-verify", Algorithm 1)
// fused with the Saguaro fan-out ("speculation cache strategy": the top-F_k
// draft tokens of every lookahead row k) over the same draft logits, so
// that every draft row is read from HBM once.
//
// Design.  One thread-block cluster takes one sequence at a time (work
// counter); the vocabulary axis of every row is cut into one slice per CTA.
// Each CTA streams its slices of the sequence's rows through a ring of
// shared-memory stages filled by TMA bulk copies, in the order
//   D_0, T_0, D_1, T_1, ..., D_gamma, T_gamma
// (D_k draft row k, T_k target row k).  A draft-row pass feeds the online
// (max, sum) of q_k and the top-F_k filter (sdv_topf.cuh) in one read; a
// target-row pass the (max, sum) of p_k, after which the cluster exchanges
// its partials through distributed shared memory and decides position k.
//
// Thread 0 is the ring's producer and runs up to the ring's depth ahead of
// the consumers.  Draft rows are always read (every row feeds the fan-out),
// so they are issued without waiting for a decision; target row k is issued
// only once position k-1 was accepted.  The ring therefore stays full
// through the decisions, and no row after the first rejection is ever read
// from the target.  At the first rejection (or after the bonus row) the
// correction norm(max(0, p_n - q_n)) or the bonus p_gamma is drawn by
// inverse CDF with plain loads over the two slices just streamed (from L2)
// while the ring keeps fetching the remaining draft rows.  Each CTA keeps
// its slice's top-F_k list per row in the workspace; at the end of the
// sequence CTA r of the cluster ranks the lists of rows k = r mod CL.
#include "sdv_device.cuh"
#include "sdv_host.cuh"
#include "sdv_ring.cuh"
#include "sdv_tma.cuh"
#include "sdv_topf.cuh"

namespace sdv {

constexpr int kFusedMaxTotal = 256;  // sum of F_k the fused kernel takes

struct FusedParams {
  const void *target;  // [B, gamma+1, V]
  const void *draft;   // [B, gamma+1, V]
  const int32_t *tokens;
  const float *uniforms;
  int B, gamma, V;
  float k2;  // log2(e) / T
  int F[SD_MAX_K + 1];
  int off[SD_MAX_K + 2];
  int total;
  int32_t *n_acc;
  int32_t *out_tokens;
  float *out_prob;
  int32_t *fan_tokens;
  float *fan_logit;
  int32_t *dev_status;
  int *queue;
  uint64_t *lists;  // [gridDim.x][2][total]: each CTA's slice lists
  int nclusters;
  int seg_bytes;
};

// Ring schedule of one CTA (thread 0 only, kept in shared memory): the
// producer's position in the row order and what the consumers have decided
// about their sequence.  Item kinds: 0 draft row D_k, 1 target row T_k,
// 2 "after T_k" (waits for the decision of position k, no chunks), 3 the
// draw's re-read of T_k (and D_k) in two-row stages.
struct Sched {
  int pseq;   // producer: sequence, -1 while waiting to learn it
  int pprev;  // the sequence before (while pseq == -1)
  int ppos, pkind;
  int dseq;     // consumers' sequence
  int decided;  // positions decided
  int final;    // the target rows ended (rejection, bonus or bad row)
  int draw;     // the final decision needs the draw's re-read
  int next;     // the sequence after dseq, -1 until known
};

// The producer's current item (thread 0's registers): the next chunk's
// source(s) and the vectors left.
struct PState {
  const char *pa, *pb;
  int prem;    // vectors left in the item
  int pstg;    // vectors per chunk (kStageVecs; kStg for the draw's pairs)
  int issued;  // chunks issued so far
};

struct FusedSmem {
  MS red[1][kWarps];
  AM ared[kWarps];
  union {  // [parity]: this CTA's partials of the position (peers read)
    MS part[2][2];
    AM apart[2];
  };
  MS mrg[2];
  AM amrg;
  MS qtmp;  // thread 0: this CTA's partial of q at the current position
  int next_seq[2];
  int gx;
  float gzt, gzd, gr;
  int kind, tok;
  MS mt, md;
  Sched sc;
  DrawSmem draw;
  TopSmem top;
};

template <int DT, int VW, bool GREEDY>
struct Fused {
  const FusedParams &p;
  const Slice &sl;
  Ring &rg;
  int nv, nch, nchd;  // vectors in the slice; chunks of a row; of the draw
  size_t rowb;

  __device__ bool d_needed(int k) const {
    return (!GREEDY && k < p.gamma) || p.F[k] > 0;
  }
  __device__ const char *row(int kind, int seq, int k) const {
    const char *base = static_cast<const char *>(kind ? p.target : p.draft);
    return base + ((size_t)seq * (p.gamma + 1) + k) * rowb;
  }
  __device__ void next_row(Sched &sc) const {  // to D_{k+1} or the next seq
    sc.pkind = 0;
    if (++sc.ppos > p.gamma) {
      sc.ppos = 0;
      sc.pprev = sc.pseq;
      sc.pseq = -1;
    }
  }
  // Move the schedule to the next item that has chunks and load it into
  // the producer's registers; false while the next item waits for a
  // decision, a sequence number or the end.  sc records the item after the
  // loaded one.  Thread 0 only.
  __device__ bool next_item(Sched &sc, PState &ps) const {
    for (;;) {
      if (sc.pseq == -1) {
        if (sc.dseq != sc.pprev || sc.next < 0) return false;
        sc.pseq = sc.next;
      }
      if (sc.pseq >= p.B) return false;
      const bool cur = sc.pseq == sc.dseq;
      const int k = sc.ppos;
      const char *ra = nullptr, *rb = nullptr;
      int stg = kStageVecs;
      if (sc.pkind == 0) {  // D_k: after every decision before k
        if (k > 0 && !(cur && (sc.decided >= k || sc.final))) return false;
        sc.pkind = 1;
        if (d_needed(k)) ra = row(0, sc.pseq, k);
      } else if (sc.pkind == 1) {  // T_k, unless the target rows ended
        if (k > 0 && sc.final) {
          next_row(sc);
          continue;
        }
        sc.pkind = 2;
        ra = row(1, sc.pseq, k);
      } else if (sc.pkind == 2) {  // wait for decision k
        if (!(cur && sc.decided > k)) return false;
        if (sc.final && sc.draw) sc.pkind = 3;
        else next_row(sc);
        continue;
      } else {  // the draw's re-read of T_k (and D_k) in two-row stages
        ra = row(1, sc.pseq, k);
        if (sc.draw == 1) rb = row(0, sc.pseq, k);
        stg = kStg;
        next_row(sc);
      }
      if (ra && nv > 0) {
        ps.pa = ra + (size_t)sl.vbeg * 16;
        ps.pb = rb ? rb + (size_t)sl.vbeg * 16 : nullptr;
        ps.prem = nv;
        ps.pstg = stg;
        return true;
      }
    }
  }
  // Issue chunks while a stage is free and the next chunk is known to be
  // needed.  Thread 0 only.
  __device__ __forceinline__ void pump(Sched &sc, PState &ps,
                                       int consumed) const {
    while (ps.issued < consumed + kStages) {
      if (ps.prem == 0 && !next_item(sc, ps)) return;
      const int cnt = min(ps.pstg, ps.prem);
      const uint32_t bytes = (uint32_t)cnt * 16u;
      const int s = ps.issued % kStages;
      fence_proxy_async();
      mbar_expect_tx(&rg.full[s], ps.pb ? 2u * bytes : bytes);
      bulk_g2s(rg.buf + (size_t)s * kStageVecs, ps.pa, bytes, &rg.full[s]);
      if (ps.pb) {
        bulk_g2s(rg.buf + (size_t)s * kStageVecs + kStg, ps.pb, bytes,
                 &rg.full[s]);
        ps.pb += bytes;
      }
      ps.pa += bytes;
      ps.prem -= cnt;
      ++ps.issued;
    }
  }
};

// One draft vector per lane: the online (max, sum) of q (DQ) and the top-F
// filter (FILT) from one read, sharing the NaN-propagating vector maximum.
template <int DT, int VW, bool DQ, bool FILT>
__device__ __forceinline__ void d_vec(MS &q, WarpFilter &wf, uint32_t *cta_th,
                                      const Raw<DT, VW> &r, bool ok, int j0,
                                      float k2) {
  float z[VW];
#pragma unroll
  for (int e = 0; e < VW; ++e)
    z[e] = ok ? elt<DT, VW>(r, e) : -__builtin_huge_valf();
  const float vmax = vmax_nan_of<VW>(z);
  if (DQ && ok) {  // (an idle lane would meet -inf * k2 + inf)
    // a NaN element leaves m alone and turns s into NaN (the row is invalid)
    if (__builtin_expect(vmax > q.m, 0)) {
      q.s *= ex2((q.m - vmax) * k2);
      q.m = vmax;
    }
    // nothing finite seen yet: offset 0 (the -inf elements weigh 0)
    const float mk = q.m > kMEmpty ? -q.m * k2 : 0.f;
    if constexpr (VW == 1) {
      q.s += ex2(fmaf(z[0], k2, mk));
    } else {
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int e = 0; e < VW; e += 2) {
        const float2 t = __ffma2_rn(make_float2(z[e], z[e + 1]),
                                    make_float2(k2, k2), make_float2(mk, mk));
        acc = __fadd2_rn(acc, make_float2(ex2(t.x), ex2(t.y)));
      }
      q.s += acc.x + acc.y;
    }
  }
  if constexpr (FILT) {
    wf.nseen = max_nan(wf.nseen, vmax);
    if (__builtin_expect(!wf.seeded, 0)) wf_seed_vec<VW>(wf, z);
    if (__builtin_expect(__any_sync(0xffffffffu, vmax >= wf.th), 0)) {
#pragma unroll
      for (int e = 0; e < VW; ++e) {
        const bool take = ok && z[e] >= wf.th;
        unsigned m = __ballot_sync(0xffffffffu, take);
        if (m == 0) continue;
        const uint64_t key = make_key(ord32(z[e]), (uint32_t)(j0 + e));
        while (m) {
          const int src = __ffs(m) - 1;
          m &= m - 1;
          wf_insert(wf, shfl64(key, src));
        }
        wf_raise(wf, cta_th);
      }
    }
  }
}

// A draft-row chunk of cn vectors at stage A (vector v0 first): warp w takes
// vectors 32 w + lane, 32 (w + kWarps) + lane, ...
template <int DT, int VW, bool DQ, bool FILT>
__device__ __forceinline__ void d_chunk(MS &q, WarpFilter &wf,
                                        uint32_t *cta_th, const uint4 *A,
                                        int v0, int cn, float k2) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (FILT) wf_sync(wf, cta_th);
  if (cn == kStageVecs) {
#pragma unroll 2
    for (int base = warp * 32; base < kStageVecs; base += kThreads) {
      const int i = base + lane;
      d_vec<DT, VW, DQ, FILT>(q, wf, cta_th, sget<DT, VW>(A, i), true,
                              (v0 + i) * VW, k2);
    }
  } else {
    for (int base = warp * 32; base < cn; base += kThreads) {
      const int i = base + lane;
      Raw<DT, VW> r{};
      if (i < cn) r = sget<DT, VW>(A, i);
      d_vec<DT, VW, DQ, FILT>(q, wf, cta_th, r, i < cn, (v0 + i) * VW, k2);
    }
  }
}

// Rank the cluster's slice lists of row k of sequence seq (read from the
// workspace) and write the row's fan-out.  Block-wide.
__device__ __noinline__ void fused_merge_row(FusedSmem &sh,
                                             const FusedParams &p,
                                             const uint64_t *cl_lists,
                                             int CL, int spar, int seq,
                                             int k) {
  const int tid = threadIdx.x;
  const int F = p.F[k], total = p.total;
  if (tid == 0) sh.top.nan = 0;
  __syncthreads();
  for (int i = tid; i < CL * F; i += kThreads) {
    const int r = i / F, j = i - r * F;
    uint64_t key =
        cl_lists[(size_t)r * 2 * total + (size_t)spar * total + p.off[k] + j];
    if (key == 1ull) {  // that slice held a NaN
      sh.top.nan = 1;
      key = 0;
    }
    sh.top.flat[i] = key;
  }
  __syncthreads();
  const int nout = rank_select(sh.top, CL * F, F);
  const int bad = sh.top.nan;
  int32_t *ot = p.fan_tokens + (size_t)seq * total + p.off[k];
  float *ol =
      p.fan_logit ? p.fan_logit + (size_t)seq * total + p.off[k] : nullptr;
  for (int i = tid; i < F; i += kThreads) {
    const bool ok = !bad && i < nout;
    ot[i] = ok ? key_idx(sh.top.out[i]) : -1;
    if (ol) ol[i] = ok ? key_val(sh.top.out[i]) : __int_as_float(0x7fc00000);
  }
  if (tid == 0 && bad) status_or(p.dev_status, SD_DEV_NONFINITE);
  __syncthreads();
}

// The draw's second attempt when the residual has zero mass: inverse CDF
// over p_n alone, read with plain loads.  Every thread of the cluster calls
// it.
template <int DT, int VW>
__device__ __noinline__ DrawOut fused_redraw(cg::cluster_group &cluster,
                                             FusedSmem &sh, float *segmass,
                                             const Slice &sl,
                                             const char *trow,
                                             const Weight &W, float u,
                                             int &par) {
  const GRow<DT, VW> ra{trow};
  cluster_total(cluster, sh.draw, segmass, sl, u, par, [&] {
    mass_pass<DT, VW>(ra, ra, false, W, sl, segmass);
  });
  return draw_pick<DT, VW>(cluster, sh.draw, segmass, ra, ra, false, W, sl);
}

// Wait for the next chunk in the ring, run f on its stage, release the
// stage and let thread 0 refill the ring.  Block-wide.
template <class Fu, class F>
__device__ __forceinline__ void consume_chunk(const Fu &fu, Ring &rg,
                                              Sched &sc, PState &ps,
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

#ifndef SDV_FUSED_MINB
#define SDV_FUSED_MINB 4
#endif

template <int DT, int VW, bool GREEDY>
__global__ void __launch_bounds__(kThreads, SDV_FUSED_MINB)
    fused_kernel(const FusedParams p) {
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ FusedSmem sh;
  __shared__ uint64_t bars[2 * kStages];
  using GR = GRow<DT, VW>;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int CL = (int)cluster.num_blocks();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = p.V, gamma = p.gamma;
  const float k2 = p.k2;
  const Slice sl = make_slice(V / VW, rank, CL);
  float *segmass = reinterpret_cast<float *>(dsm);
  Ring rg;
  rg.buf = reinterpret_cast<uint4 *>(dsm + p.seg_bytes);
  rg.full = bars;
  rg.empty = bars + kStages;
  rg.dev_status = p.dev_status;
  const int nv = sl.vend - sl.vbeg;
  const Fused<DT, VW, GREEDY> fu{p, sl, rg, nv,
                                 (nv + kStageVecs - 1) / kStageVecs,
                                 (nv + kStg - 1) / kStg,
                                 (size_t)V * elt_bytes<DT>()};
  uint64_t *mylist = p.lists + (size_t)blockIdx.x * 2 * p.total;
  const uint64_t *cl_lists = p.lists + (size_t)(blockIdx.x - rank) * 2 * p.total;

  int seq = (int)(blockIdx.x / CL);
  if (tid == 0) {
    sh.top.th = 0;
    sh.sc = Sched{seq, -1, 0, 0, seq, 0, 0, 0, -1};
  }
  ring_init(rg);  // (a block barrier)
  int par = 0, spar = 0, consumed = 0;
  uint32_t phase = 0;
  PState ps{nullptr, nullptr, 0, 0, 0};
  if (tid == 0) fu.pump(sh.sc, ps, consumed);

  auto consume = [&](auto &&f) {
    consume_chunk(fu, rg, sh.sc, ps, consumed, phase, p.dev_status, f);
  };

  while (seq < p.B) {
    if (rank == 0 && tid == 0)
      sh.next_seq[spar] = p.nclusters + atomicAdd(p.queue, 1);
    bool final = false;
    int bad_token = 0;
    for (int k = 0; k <= gamma; ++k) {
      // ---------------- draft row: q_k statistics and top-F_k ------------
      const int F = p.F[k];
      if (fu.d_needed(k)) {
        const bool dq = !GREEDY && k < gamma;
        MS q = ms_empty();
        WarpFilter wf;
        wf_init(wf, F > 0 ? F : 1);
        for (int c = 0; c < fu.nch; ++c) {
          const int v0 = sl.vbeg + c * kStageVecs;
          const int cn = min(kStageVecs, nv - c * kStageVecs);
          consume([&](const uint4 *A) {
            if (c == 0 && F > 0) {
              // seed every warp's threshold from the whole first chunk: the
              // CTA takes the largest value that F lane maxima of one warp
              // reach, so the warps start from a common high threshold
              float m1 = -__builtin_huge_valf(), m2 = -__builtin_huge_valf();
              for (int base = warp * 32; base < cn; base += kThreads) {
                const int i = base + lane;
                if (i < cn) {
                  const Raw<DT, VW> r = sget<DT, VW>(A, i);
#pragma unroll
                  for (int e = 0; e < VW; ++e) top2_add(m1, m2, elt<DT, VW>(r, e));
                }
              }
              wf_seed2(wf, m1, m2);
              if (lane == 0 && wf.th > -__builtin_huge_valf())
                atomicMax(&sh.top.th, ord32(wf.th));
              __syncthreads();
            }
            if (dq && F > 0) d_chunk<DT, VW, true, true>(q, wf, &sh.top.th, A, v0, cn, k2);
            else if (dq) d_chunk<DT, VW, true, false>(q, wf, &sh.top.th, A, v0, cn, k2);
            else d_chunk<DT, VW, false, true>(q, wf, &sh.top.th, A, v0, cn, k2);
          });
        }
        if (dq) {
          MS qa[1] = {q};
          block_reduce_ms<1>(qa, k2, sh.red);
          if (tid == 0) sh.qtmp = qa[0];
        }
        if (F > 0) {
          const int anynan = __syncthreads_or(wf.nseen != wf.nseen);
          wf_export(wf, sh.top);
          __syncthreads();
          const int nout = rank_select(sh.top, kWarps * F, F);
          uint64_t *dst = mylist + (size_t)spar * p.total + p.off[k];
          for (int i = tid; i < F; i += kThreads)
            dst[i] = anynan ? (i == 0 ? 1ull : 0ull)
                            : (i < nout ? sh.top.out[i] : 0ull);
          if (tid == 0) sh.top.th = 0;
        }
        __syncthreads();
      }
      if (final) continue;

      // ---------------- target row: p_k statistics, decision -------------
      // this position's gathers: loaded now (warp 1), stored after the row
      int gx = -1;
      float gzt = 0.f, gzd = 0.f, gr = 0.f;
      const bool gath = tid == 32 && k < gamma;
      if (gath) {
        gx = p.tokens[(size_t)seq * gamma + k];
        if (!GREEDY) {
          if (gx >= 0 && gx < V) {
            gzt = load_logit<DT>(fu.row(1, seq, k), gx);
            gzd = load_logit<DT>(fu.row(0, seq, k), gx);
          }
          gr = p.uniforms[(size_t)seq * (gamma + 1) + k];
        }
      }
      MS pst = ms_empty();
      AM am = am_empty();
      for (int c = 0; c < fu.nch; ++c) {
        const int v0 = sl.vbeg + c * kStageVecs;
        const int cn = min(kStageVecs, nv - c * kStageVecs);
        consume([&](const uint4 *A) {
          for (int i = tid; i < cn; i += kThreads) {
            if constexpr (GREEDY) am_add<DT, VW>(am, sget<DT, VW>(A, i), (v0 + i) * VW);
            else ms_add<DT, VW>(pst, sget<DT, VW>(A, i), k2);
          }
        });
      }
      if (gath) {
        sh.gx = gx;
        sh.gzt = gzt;
        sh.gzd = gzd;
        sh.gr = gr;
      }
      if constexpr (GREEDY) {
        am = block_reduce_am(am, sh.ared);
        if (tid == 0) sh.apart[par] = am;
      } else {
        MS pa[1] = {pst};
        block_reduce_ms<1>(pa, k2, sh.red);
        if (tid == 0) {
          sh.part[par][0] = pa[0];
          sh.part[par][1] = k < gamma ? sh.qtmp : ms_empty();
        }
      }
      cluster.sync();
      if (warp < (GREEDY ? 1 : 2)) {  // every CTA merges in rank order
        if constexpr (GREEDY) {
          AM a = am_empty();
          if (lane < CL) a = cluster.map_shared_rank(&sh, lane)->apart[par];
          a = warp_down_am(a);
          if (lane == 0) sh.amrg = a;
        } else {
          MS m = ms_empty();
          if (lane < CL) m = cluster.map_shared_rank(&sh, lane)->part[par][warp];
          m = warp_down_ms(m, k2);
          if (lane == 0) sh.mrg[warp] = m;
        }
      }
      __syncthreads();
      par ^= 1;
      if (tid == 0) {  // the accept test of position k
        const int x = sh.gx;
        const bool bad = k < gamma && (x < 0 || x >= V);
        bool invalid, acc = false;
        int kind = 0;
        if constexpr (GREEDY) {
          const AM a = sh.amrg;
          invalid = a.bad || !(a.v > -kInf);
          acc = !invalid && k < gamma && x == a.i;
          sh.tok = a.i;
        } else {
          const MS mt = sh.mrg[0], md = sh.mrg[1];
          invalid = !ms_valid(mt) || (k < gamma && !ms_valid(md));
          if (!invalid && k < gamma && !bad) {
            const float rho = accept_ratio(sh.gzt, sh.gzd, mt, md, k2);
            acc = sh.gr <= rho;
          }
          sh.mt = mt;
          sh.md = md;
        }
        if (invalid) kind = 3;
        else if (k == gamma) kind = 2;
        else if (!acc) kind = 1;
        sh.kind = kind | (bad ? 4 : 0);
        Sched &sc = sh.sc;
        sc.decided = k + 1;
        if (kind) {
          sc.final = 1;
          sc.draw = (!GREEDY && kind != 3) ? kind : 0;
        }
        if (k == 0) sc.next = cluster.map_shared_rank(&sh, 0)->next_seq[spar];
        fu.pump(sc, ps, consumed);
      }
      __syncthreads();
      const int kind = sh.kind & 3;
      bad_token |= sh.kind >> 2;
      if (!kind) continue;
      final = true;
      const int n = k;
      // ---------------- outputs of the verify ----------------------------
      if (kind == 3) {  // unusable row: outputs -1
        if (rank == 0) {
          for (int t = tid; t <= gamma; t += kThreads)
            p.out_tokens[(size_t)seq * (gamma + 1) + t] = -1;
          if (tid == 0) {
            p.n_acc[seq] = -1;
            if (p.out_prob) p.out_prob[seq] = 0.f;
            status_or(p.dev_status,
                      SD_DEV_NONFINITE | (bad_token ? SD_DEV_BAD_TOKEN : 0));
          }
        }
      } else if (GREEDY) {
        if (rank == 0) {
          const int tk = sh.tok;
          for (int t = tid; t <= gamma; t += kThreads) {
            int v = -1;
            if (t < n) v = p.tokens[(size_t)seq * gamma + t];
            else if (t == n) v = tk;
            p.out_tokens[(size_t)seq * (gamma + 1) + t] = v;
          }
          if (tid == 0) {
            p.n_acc[seq] = n;
            if (p.out_prob) p.out_prob[seq] = 1.f;
            status_or(p.dev_status, bad_token ? SD_DEV_BAD_TOKEN : 0);
          }
        }
      } else {
        // correction (kind 1) or bonus (kind 2) by inverse CDF: the slices
        // of position n stream through the ring again (from L2) in
        // two-row stages; the segment masses land in segmass
        const bool has_q = kind == 1;
        Weight W;
        W.k2 = k2;
        W.mtk = sh.mt.m * k2;
        W.ist = 1.f / sh.mt.s;
        W.mdk = sh.md.m * k2;
        W.cq = 1.f / sh.md.s;
        const float u = p.uniforms[(size_t)seq * (gamma + 1) + gamma];
        cluster_total(cluster, sh.draw, segmass, sl, u, par, [&] {
          for (int c = 0; c < fu.nchd; ++c) {
            const int cn = min(kStg, nv - c * kStg);
            consume([&](const uint4 *A) {
              const uint4 *Bq = A + kStg;
              for (int g = warp; g * 32 < cn; g += kWarps) {  // warp-uniform
                const int i = g * 32 + lane;
                float acc = 0.f;
                if (i < cn) {
                  float w[VW];
                  weights<DT, VW>(sget<DT, VW>(A, i),
                                  sget<DT, VW>(has_q ? Bq : A, i), has_q, W, w);
#pragma unroll
                  for (int e = 0; e < VW; ++e) acc += w[e];
                }
                acc = warp_down_sum(acc);
                if (lane == 0) segmass[c * (kStg / 32) + g] = acc;
              }
            });
          }
        });
        const GR ra{fu.row(1, seq, n)};
        const GR rb{has_q ? fu.row(0, seq, n) : fu.row(1, seq, n)};
        DrawOut o = draw_pick<DT, VW>(cluster, sh.draw, segmass, ra, rb, has_q,
                                      W, sl);
        int zero_mass = 0;
        if (o.owner < 0) {  // residual of zero mass: draw from p_n instead
          zero_mass = 1;
          __syncthreads();
          o = fused_redraw<DT, VW>(cluster, sh, segmass, sl, fu.row(1, seq, n),
                                   W, u, par);
        }
        if (o.owner == rank && warp == 0) {
          for (int t = lane; t <= gamma; t += 32) {
            int v = -1;
            if (t < n) v = p.tokens[(size_t)seq * gamma + t];
            else if (t == n) v = o.t;
            p.out_tokens[(size_t)seq * (gamma + 1) + t] = v;
          }
          if (lane == 0) {
            p.n_acc[seq] = n;
            if (p.out_prob) p.out_prob[seq] = (float)((double)o.wt / o.N);
            status_or(p.dev_status, (bad_token ? SD_DEV_BAD_TOKEN : 0) |
                                        (zero_mass ? SD_DEV_ZERO_MASS : 0));
          }
        }
        __syncthreads();
      }
    }

    // ---------------- fan-out: rank the CTAs' lists of each row -----------
    __threadfence();
    cluster.sync();
    for (int k = rank; k <= gamma; k += CL)  // CTA-uniform
      if (p.F[k] > 0) fused_merge_row(sh, p, cl_lists, CL, spar, seq, k);
    // next sequence (rank 0 published it before this sequence's first sync)
    seq = cluster.map_shared_rank(&sh, 0)->next_seq[spar];
    spar ^= 1;
    if (tid == 0) {
      Sched &sc = sh.sc;
      sc.dseq = seq;
      sc.decided = 0;
      sc.final = 0;
      sc.draw = 0;
      sc.next = -1;
      fu.pump(sc, ps, consumed);
    }
    __syncthreads();
  }
  cluster.sync();  // no CTA leaves while a peer may still read its smem
}

using FusedKernel = void (*)(const FusedParams);

static FusedKernel pick_fused(int dt, bool greedy) {
  if (dt == SD_F32)
    return greedy ? fused_kernel<0, 4, true> : fused_kernel<0, 4, false>;
  return greedy ? fused_kernel<1, 8, true> : fused_kernel<1, 8, false>;
}

static size_t fused_lists_bytes(int sms) {
  return (size_t)sms * 4 * 2 * kFusedMaxTotal * sizeof(uint64_t);
}

sd_status linear_launch(const void *target, const void *draft, sd_dtype dt,
                        long long d_seq_rows, const int32_t *tokens,
                        const float *uniforms, int B, int gamma, int V,
                        float T, int32_t *n_acc, int32_t *out_tokens,
                        float *out_prob, float *out_accept, float *out_resid,
                        int32_t *dev_status, void *ws, size_t ws_bytes,
                        cudaStream_t stream);

}  // namespace sdv

extern "C" size_t sd_verify_linear_fanout_workspace(int B, int gamma, int V,
                                                    sd_dtype dt) {
  int sms = 0;
  if (sdv::check_device(&sms) != SD_OK) sms = 256;
  const size_t a = 256 + sdv::fused_lists_bytes(sms);
  const size_t b = sd_verify_linear_workspace(B, gamma, V, dt);
  return a > b ? a : b;
}

extern "C" sd_status sd_verify_linear_fanout(
    const void *target_logits, const void *draft_logits, sd_dtype dt,
    const int32_t *draft_tokens, const float *uniforms, int B, int gamma,
    int V, float T, const int32_t *F, int32_t *n_accepted,
    int32_t *out_tokens, float *out_prob, int32_t *fan_tokens,
    float *fan_logit, int32_t *dev_status, void *workspace, size_t ws_bytes,
    void *stream) {
  using namespace sdv;
  SDV_REQUIRE(dt == SD_F32 || dt == SD_BF16, "bad dtype %d", (int)dt);
  SDV_REQUIRE(B >= 0, "B < 0");
  SDV_REQUIRE(gamma >= 0 && gamma <= SD_MAX_K, "gamma=%d outside [0, %d]",
              gamma, SD_MAX_K);
  SDV_REQUIRE(V >= 1 && V <= SD_MAX_V, "V=%d outside [1, %d]", V, SD_MAX_V);
  SDV_REQUIRE(T >= 0.f && std::isfinite(T), "T must be finite and >= 0");
  SDV_REQUIRE(F != nullptr, "F is null");
  int total = 0, maxF = 0;
  for (int k = 0; k <= gamma; ++k) {
    SDV_REQUIRE(F[k] >= 0, "F[%d] < 0", k);
    if (F[k] > SD_MAX_FANOUT || F[k] > V)
      return fail(SD_ERR_UNSUPPORTED, "F[%d]=%d exceeds min(V, %d)", k, F[k],
                  SD_MAX_FANOUT);
    total += F[k];
    maxF = F[k] > maxF ? F[k] : maxF;
  }
  if (B == 0) return SD_OK;
  SDV_REQUIRE(target_logits && draft_logits && n_accepted && out_tokens,
              "null pointer");
  SDV_REQUIRE(total == 0 || fan_tokens, "fan_tokens is null");
  SDV_REQUIRE(gamma == 0 || draft_tokens, "draft_tokens is null");
  SDV_REQUIRE(T == 0.f || uniforms, "uniforms is null");
  int sms = 0;
  sd_status st = check_device(&sms);
  if (st != SD_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool greedy = (T == 0.f);
  const int eb = dt == SD_F32 ? 4 : 2, vw = dt == SD_F32 ? 4 : 8;
  const bool vec = aligned16(target_logits) && aligned16(draft_logits) &&
                   ((size_t)V * eb) % 16 == 0;
  const long long nvec = V / vw;
  FusedKernel kern = pick_fused(dt, greedy);
  auto smem_for = [&](int cl) {
    const long long per_cta = (nvec + cl - 1) / cl;
    const size_t seg = ((size_t)((per_cta + 31) / 32) * 4 + 127) / 128 * 128;
    return seg + (size_t)kRingBytes;
  };
  // the largest cluster at which all B sequences are resident at once (a
  // slice of at least one full stage per CTA; CL * max F keys gathered in
  // one merge), else single CTAs taking sequences from the work counter
  int CL = 1, maxc = 0;
  const int forced = tune(SD_TUNE_CLUSTER);
  for (int c = 16; c >= 1; c /= 2) {
    if (forced && c != forced && c != 1) continue;
    if (c > 1 && nvec / c < kStageVecs && !forced) continue;
    if (c * maxF > kWarps * SD_MAX_FANOUT) continue;
    int mc = 0;
    st = max_active_clusters((const void *)kern, c, smem_for(c), &mc);
    if (st != SD_OK) return st;
    if (B <= mc || c == 1 || forced) {
      CL = c;
      maxc = mc;
      break;
    }
  }
  const size_t smem = smem_for(CL);
  const size_t seg_bytes = smem - kRingBytes;
  const bool fused = vec && total > 0 && total <= kFusedMaxTotal &&
                     kStg % 32 == 0 &&
                     smem <= 64 * 1024 && maxc > 0 &&
                     tune(SD_TUNE_FUSED) != 0;
  if (!fused) {
    // the two calls one after the other (same results)
    st = linear_launch(target_logits, draft_logits, dt, gamma + 1,
                       draft_tokens, uniforms, B, gamma, V, T, n_accepted,
                       out_tokens, out_prob, nullptr, nullptr, dev_status,
                       workspace, ws_bytes, s);
    if (st != SD_OK) return st;
    return sd_fanout_topk(draft_logits, dt, B, gamma, V, F, fan_tokens,
                          fan_logit, dev_status, nullptr, 0, stream);
  }
  const int nclusters = B < maxc ? B : maxc;
  const size_t need = 256 + (size_t)nclusters * CL * 2 * total * sizeof(uint64_t);
  if (!workspace || ws_bytes < need)
    return fail(SD_ERR_INVALID_ARG, "workspace of >= %zu bytes required", need);
  FusedParams prm;
  prm.target = target_logits;
  prm.draft = draft_logits;
  prm.tokens = draft_tokens;
  prm.uniforms = uniforms;
  prm.B = B;
  prm.gamma = gamma;
  prm.V = V;
  prm.k2 = greedy ? 0.f : (float)(1.4426950408889634 / (double)T);
  int o = 0;
  for (int k = 0; k <= gamma; ++k) {
    prm.F[k] = F[k];
    prm.off[k] = o;
    o += F[k];
  }
  prm.off[gamma + 1] = o;
  prm.total = total;
  prm.n_acc = n_accepted;
  prm.out_tokens = out_tokens;
  prm.out_prob = out_prob;
  prm.fan_tokens = fan_tokens;
  prm.fan_logit = fan_logit;
  prm.dev_status = dev_status;
  prm.queue = static_cast<int *>(workspace);
  prm.lists = reinterpret_cast<uint64_t *>(static_cast<char *>(workspace) + 256);
  prm.nclusters = nclusters;
  prm.seg_bytes = (int)seg_bytes;
  SDV_CUDA(cudaMemsetAsync(workspace, 0, sizeof(int), s));
  void *args[] = {&prm};
  return launch_clusters((const void *)kern, nclusters, CL, smem, s, args);
}
