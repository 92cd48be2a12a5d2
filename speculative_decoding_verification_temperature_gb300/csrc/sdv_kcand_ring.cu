// sdv_kcand_ring.cu -- K-candidate verify with verifier self-selection
// (SpecDiff-2, "core method"), streaming version for 16-byte aligned rows.
//
// One thread-block cluster verifies one sequence b at a time; the
// vocabulary axis of every row is cut into one slice per CTA.  Position j
// is one step over the rows it needs: the shared draft-marginal row (b, j)
// and the target row (b, k, j) of every candidate k still alive.  Each CTA
// streams its slices of those rows back to back through a ring of
// shared-memory stages filled by TMA bulk copies (thread 0 issues them, up
// to the ring's depth ahead), keeping one online (max, sum) per thread and
// folding it into per-warp partials at the end of each row.  The cluster
// then exchanges the rows' partials through distributed shared memory and
// warp 0 applies the accept test r <= p(x)/q(x) of each live candidate.
// The next position's rows are issued once its live set is known, so no
// row after a candidate's first rejection is read.  The candidate with the
// most accepted tokens (lowest k on ties) gets the correction (its
// rejection pair streamed again, from L2) or the bonus (its row gamma) by
// the cluster-wide inverse-CDF draw.
#include "sdv_device.cuh"
#include "sdv_host.cuh"
#include "sdv_ring.cuh"
#include "sdv_tma.cuh"

namespace sdv {

struct KRParams {
  const void *target;  // [B, K, gamma+1, V]
  const void *draft;   // [B, gamma, V]
  const int32_t *tokens;    // [B, K, gamma]
  const float *uniforms;    // [B, K, gamma+1]
  int B, K, gamma, V;
  float k2;
  int32_t *n_acc, *sel_k, *out_tokens, *n_per_cand;
  float *out_prob;
  int32_t *dev_status;
  int *queue;
  int nclusters;
  int seg_bytes;
  // Helping (sampled rows; all null when off).  A cluster whose sequence is
  // done computes rows of positions ahead of the scans still running: each
  // CTA claims a position of a running sequence for its rank, streams its
  // slice of the position's draft-marginal row and of the target rows of
  // the candidates alive at the claim, with the owner's own code (hence the
  // same bits), stores each row's partial and raises its flag.  An owner CTA
  // reads the flags of the next position's rows when it decides, and its
  // producer skips the rows found done.  Nobody waits on a flag.
  int *helping;   // set once a cluster has started helping
  int *active;    // [nclusters]: sequence + 1 being verified, or 0
  int *opos;      // [B]: the owner's next position
  int *oalive;    // [B]: its live candidates
  int *hpos;      // [B][kHelpRanks]: next (position, row) to hand to a
                  // helper, as position * (K + 1) + row
  int *hflag;     // [B][gamma][K+1][kHelpRanks]: partial published
  float2 *hpart;  // [B][gamma][K+1][kHelpRanks]: (m, s)
};

constexpr int kKRows = SD_MAX_K + 1;  // draft row + one per candidate
constexpr int kHelpRanks = 16;        // record stride: the largest cluster


// Ring schedule (thread 0 only, in shared memory).  Producer item kinds:
// 0 the draft row of position pj, 1 the target rows of its live candidates
// (next candidate pk), 2 wait for decision pj, 3 after the scan (the draw's
// pair, or the bonus row), 4 wait for the bonus row's exchange (then its
// draw), 5 sequence done.
struct KSched {
  int pseq, pprev, pj, pkind, pk;
  int dseq;      // consumers' sequence
  int decided;   // positions decided
  unsigned alive;  // live candidates after the last decision
  int done;      // the scan is over
  int fkind;     // after the scan: 0 nothing, 1 residual pair, 2 bonus row
  int ksel, nsel;
  int bdone;     // bonus row exchanged: 1 valid, 2 unusable
  int next;      // the sequence after dseq, -1 until known
  unsigned skip;  // rows of position pj done by helpers: bit 0 the draft
                  // row, bit 1 + k candidate k's target row
};

// The producer's current item (thread 0's registers).
struct KPState {
  const char *pa, *pb;
  int prem, pstg, issued;
};

struct KRSmem {
  union {  // this position's per-warp partials, by row
    MS wpart[kKRows][kWarps];
    AM wapart[kKRows][kWarps];
  };
  union {  // [parity][row]: this CTA's partials (peers read)
    MS part[2][kKRows];
    AM apart[2][kKRows];
  };
  union {
    MS mrg[kKRows];
    AM amrg[kKRows];
  };
  int gx[SD_MAX_K];
  float gzt[SD_MAX_K], gzd[SD_MAX_K], gr[SD_MAX_K];
  int n_k[SD_MAX_K];
  MS rej_t[SD_MAX_K], rej_d[SD_MAX_K];  // stats at the rejection position
  int rej_am[SD_MAX_K];                 // greedy: argmax there
  unsigned alive;
  int invalid, bad_token;
  int next_seq[2];
  KSched sc;
  DrawSmem draw;
  MS hv[kKRows];  // helpers' partials of the next position's rows
  int hs, hj, hr;  // a helper's claim: sequence, position, row
  int hseen;      // the helping flag, read at the position's start
};

template <int DT, int VW, bool GREEDY>
struct KFu {
  const KRParams &p;
  const Slice &sl;
  Ring &rg;
  int nv;
  size_t rowb;

  __device__ unsigned full() const {
    return p.K >= 32 ? 0xffffffffu : ((1u << p.K) - 1u);
  }
  __device__ const char *trow(int b, int k, int j) const {
    return static_cast<const char *>(p.target) +
           (((size_t)b * p.K + k) * (p.gamma + 1) + j) * rowb;
  }
  __device__ const char *drow(int b, int j) const {
    return static_cast<const char *>(p.draft) +
           ((size_t)b * p.gamma + j) * rowb;
  }
  __device__ bool next_item(KSched &sc, KPState &ps) const {
    for (;;) {
      if (sc.pseq == -1) {
        if (sc.dseq != sc.pprev || sc.next < 0) return false;
        sc.pseq = sc.next;
      }
      if (sc.pseq >= p.B) return false;
      const bool cur = sc.pseq == sc.dseq;
      const int j = sc.pj, b = sc.pseq;
      const char *ra = nullptr, *rb = nullptr;
      int stg = kStageVecs;
      if (sc.pkind == 0) {  // draft row of position j (after decision j-1)
        if (j >= p.gamma) {
          sc.pkind = 3;
          continue;
        }
        sc.pkind = 1;
        sc.pk = 0;
        if (!GREEDY && !(sc.skip & 1u)) ra = drow(b, j);
      } else if (sc.pkind == 1) {  // target rows of the live candidates
        const unsigned alive = (j == 0 ? full() : sc.alive) & ~(sc.skip >> 1);
        int k = sc.pk;
        while (k < p.K && !(alive >> k & 1u)) ++k;
        if (k >= p.K) {
          sc.pkind = 2;
          continue;
        }
        sc.pk = k + 1;
        ra = trow(b, k, j);
      } else if (sc.pkind == 2) {  // wait for decision j
        if (!(cur && sc.decided > j)) return false;
        if (sc.done) {
          sc.pkind = 3;
        } else {
          sc.pj = j + 1;
          sc.pkind = 0;
        }
        continue;
      } else if (sc.pkind == 3) {  // after the scan
        if (!(cur && sc.done)) return false;
        if (sc.fkind == 1) {
          ra = trow(b, sc.ksel, sc.nsel);
          rb = drow(b, sc.nsel);
          stg = kStg;
          sc.pkind = 5;
        } else if (sc.fkind == 2) {
          ra = trow(b, sc.ksel, p.gamma);
          sc.pkind = 4;
        } else {
          sc.pkind = 5;
          continue;
        }
      } else if (sc.pkind == 4) {  // the bonus row's draw
        if (!(cur && sc.bdone)) return false;
        sc.pkind = 5;
        if (GREEDY || sc.bdone != 1) continue;
        ra = trow(b, sc.ksel, p.gamma);
        stg = kStg;
      } else {  // sequence done
        sc.pprev = sc.pseq;
        sc.pseq = -1;
        sc.pj = 0;
        sc.pkind = 0;
        sc.skip = 0;
        continue;
      }
      if (ra && nv > 0) {  // (greedy reads no draft row)
        ps.pa = ra + (size_t)sl.vbeg * 16;
        ps.pb = rb ? rb + (size_t)sl.vbeg * 16 : nullptr;
        ps.prem = nv;
        ps.pstg = stg;
        return true;
      }
    }
  }
  __device__ __forceinline__ void pump(KSched &sc, KPState &ps,
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
  // Thread 0, after the decision that ended the scan: the selection and
  // what to read next.
  __device__ void end_scan(KSched &sc, const KRSmem &sh) const {
    sc.done = 1;
    int nsel = -1, ksel = 0;
    for (int k = 0; k < p.K; ++k)
      if (sh.n_k[k] > nsel) {
        nsel = sh.n_k[k];
        ksel = k;
      }
    sc.ksel = ksel;
    sc.nsel = nsel;
    if (sh.invalid) sc.fkind = 0;
    else if (nsel == p.gamma) sc.fkind = 2;
    else sc.fkind = GREEDY ? 0 : 1;
  }
};

template <class Fu, class F>
__device__ __forceinline__ void kr_consume(const Fu &fu, Ring &rg,
                                           KSched &sc, KPState &ps,
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

// Zero residual mass: draw from p alone, read with plain loads.
template <int DT, int VW>
__device__ __noinline__ DrawOut kr_redraw(cg::cluster_group &cluster,
                                          KRSmem &sh, float *segmass,
                                          const Slice &sl, const char *trow,
                                          const Weight &W, float u,
                                          int &par) {
  const GRow<DT, VW> ra{trow};
  cluster_total(cluster, sh.draw, segmass, sl, u, par, [&] {
    mass_pass<DT, VW>(ra, ra, false, W, sl, segmass);
  });
  return draw_pick<DT, VW>(cluster, sh.draw, segmass, ra, ra, false, W, sl);
}

template <int DT, int VW, bool GREEDY>
__global__ void __launch_bounds__(kThreads, 4)
    kcand_ring_kernel(const KRParams p) {
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ KRSmem sh;
  __shared__ uint64_t bars[2 * kStages];
  using GR = GRow<DT, VW>;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int CL = (int)cluster.num_blocks();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = p.V, K = p.K, gamma = p.gamma, G1 = gamma + 1;
  const float k2 = p.k2;
  const Slice sl = make_slice(V / VW, rank, CL);
  float *segmass = reinterpret_cast<float *>(dsm);
  Ring rg;
  rg.buf = reinterpret_cast<uint4 *>(dsm + p.seg_bytes);
  rg.full = bars;
  rg.empty = bars + kStages;
  rg.dev_status = p.dev_status;
  const int nv = sl.vend - sl.vbeg;
  const int nch = (nv + kStageVecs - 1) / kStageVecs;
  const int nchd = (nv + kStg - 1) / kStg;
  const KFu<DT, VW, GREEDY> fu{p, sl, rg, nv, (size_t)V * elt_bytes<DT>()};
  const unsigned full = fu.full();

  int b = (int)(blockIdx.x / CL);
  if (tid == 0) {
    KSched &sc = sh.sc;
    sc.pseq = b;
    sc.pprev = -1;
    sc.pj = 0;
    sc.pkind = 0;
    sc.pk = 0;
    sc.dseq = b;
    sc.decided = 0;
    sc.alive = full;
    sc.done = 0;
    sc.fkind = 0;
    sc.ksel = sc.nsel = 0;
    sc.bdone = 0;
    sc.next = -1;
    sc.skip = 0;
  }
  ring_init(rg);  // (a block barrier)
  int par = 0, seqpar = 0, consumed = 0;
  uint32_t phase = 0;
  KPState ps{nullptr, nullptr, 0, 0, 0};
  auto consume = [&](auto &&f) {
    kr_consume(fu, rg, sh.sc, ps, consumed, phase, p.dev_status, f);
  };
  // One row through the ring: per-thread online state, folded into the
  // per-warp partial of row r at the end.
  auto stream_row = [&](int r) {
    MS st = ms_empty();
    AM am = am_empty();
    for (int c = 0; c < nch; ++c) {
      const int v0 = sl.vbeg + c * kStageVecs;
      const int cn = min(kStageVecs, nv - c * kStageVecs);
      consume([&](const uint4 *A) {
        for (int i = tid; i < cn; i += kThreads) {
          if constexpr (GREEDY) am_add<DT, VW>(am, sget<DT, VW>(A, i), (v0 + i) * VW);
          else ms_add<DT, VW>(st, sget<DT, VW>(A, i), k2);
        }
      });
    }
    if constexpr (GREEDY) {
      am = warp_down_am(am);
      if (lane == 0) sh.wapart[r][warp] = am;
    } else {
      st = warp_down_ms(st, k2);
      if (lane == 0) sh.wpart[r][warp] = st;
    }
  };
  // Fold the per-warp partials of rows [0, nrows) into this CTA's slot,
  // exchange over the cluster and merge in rank order into mrg.
  auto exchange = [&](int nrows, int spar) {
    __syncthreads();
    if (tid < nrows) {
      if constexpr (GREEDY) {
        AM a = sh.wapart[tid][0];
        for (int w = 1; w < kWarps; ++w) a = am_merge(a, sh.wapart[tid][w]);
        sh.apart[par][tid] = a;
      } else {
        MS a = sh.wpart[tid][0];
        for (int w = 1; w < kWarps; ++w) a = ms_merge(a, sh.wpart[tid][w], k2);
        sh.part[par][tid] = a;
      }
    }
    cluster.sync();
    for (int r = warp; r < nrows; r += kWarps) {
      if constexpr (GREEDY) {
        AM a = am_empty();
        if (lane < CL) a = cluster.map_shared_rank(&sh, lane)->apart[par][r];
        a = warp_down_am(a);
        if (lane == 0) sh.amrg[r] = a;
      } else {
        MS m = ms_empty();
        if (lane < CL) m = cluster.map_shared_rank(&sh, lane)->part[par][r];
        m = warp_down_ms(m, k2);
        if (lane == 0) sh.mrg[r] = m;
      }
    }
    if (tid == 0 && sh.sc.next < 0)
      sh.sc.next = cluster.map_shared_rank(&sh, 0)->next_seq[spar];
    __syncthreads();
    par ^= 1;
  };

  // a helper's row r: this CTA's partial, as the owner's exchange folds it
  auto take_row = [&](int r, int row) {
    if (tid == 0) {
      sh.wpart[r][0] = sh.hv[row];
      for (int w = 1; w < kWarps; ++w) sh.wpart[r][w] = ms_empty();
    }
  };
  const bool help = !GREEDY && p.hflag != nullptr;
  const int cid = (int)(blockIdx.x / CL);
  auto hrec = [&](int s, int j, int row) {
    return (((size_t)s * gamma + j) * (K + 1) + row) * kHelpRanks + rank;
  };

  if (tid == 0) fu.pump(sh.sc, ps, consumed);
  while (b < p.B) {
    if (help && tid == 0 && rank == 0) {
      st_relaxed_gpu(p.opos + b, 0);
      st_relaxed_gpu(p.oalive + b, (int)full);
      st_relaxed_gpu(p.active + cid, b + 1);
    }
    if (tid == 0) {
      if (rank == 0)
        sh.next_seq[seqpar] = p.nclusters + atomicAdd(p.queue, 1);
      sh.alive = full;
      sh.invalid = 0;
      sh.bad_token = 0;
    }
    if (tid < K) sh.n_k[tid] = gamma;
    __syncthreads();
    if (gamma == 0) {  // no position: the bonus of k = 0
      if (tid == 0) {
        fu.end_scan(sh.sc, sh);
        fu.pump(sh.sc, ps, consumed);
      }
      __syncthreads();
    }
    // ---------------- scan positions while a candidate is alive ----------
    for (int j = 0; j < gamma; ++j) {
      const unsigned alive = sh.alive;
      // gathers for the accept tests (warp 1), stored after the rows
      const int gk = tid - 32;
      const bool gath = gk >= 0 && gk < K && (alive >> gk & 1u);
      int gx = -1;
      float gzt = 0.f, gzd = 0.f, gru = 0.f;
      if (gath) {
        gx = p.tokens[((size_t)b * K + gk) * gamma + j];
        if (!GREEDY) {
          if (gx >= 0 && gx < V) {
            gzt = load_logit<DT>(fu.trow(b, gk, j), gx);
            gzd = load_logit<DT>(fu.drow(b, j), gx);
          }
          gru = p.uniforms[((size_t)b * K + gk) * G1 + j];
        }
      }
      // rows that helpers did for this CTA's slice are taken, not streamed;
      // the helping flag is read here, for the decision after the exchange
      const unsigned skip = help ? sh.sc.skip : 0u;
      if (help && tid == 64) sh.hseen = ld_relaxed_gpu(p.helping);
      int r = 0;
      if (!GREEDY) {
        if (skip & 1u) take_row(r++, 0);
        else stream_row(r++);
      }
      for (int k = 0; k < K; ++k)
        if (alive >> k & 1u) {
          if (skip >> (1 + k) & 1u) take_row(r++, 1 + k);
          else stream_row(r++);
        }
      if (gath) {
        sh.gx[gk] = gx;
        sh.gzt[gk] = gzt;
        sh.gzd[gk] = gzd;
        sh.gr[gk] = gru;
      }
      exchange(r, seqpar);
      if (warp == 0) {  // accept tests, one lane per live candidate
        bool acc = false, bad = false, inv = false;
        const int k = lane;
        if (k < K && (alive >> k & 1u)) {
          const int rk = (GREEDY ? 0 : 1) + __popc(alive & ((1u << k) - 1u));
          const int x = sh.gx[k];
          bad = x < 0 || x >= V;
          if constexpr (GREEDY) {
            const AM a = sh.amrg[rk];
            inv = a.bad || !(a.v > -kInf);
            acc = !inv && x == a.i;
            if (!acc) sh.rej_am[k] = a.i;
          } else {
            const MS mt = sh.mrg[rk], md = sh.mrg[0];
            inv = !ms_valid(mt) || !ms_valid(md);
            if (!inv && !bad) {
              const float rho =
                  accept_ratio(sh.gzt[k], sh.gzd[k], mt, md, k2);
              acc = sh.gr[k] <= rho;
            }
            if (!acc) {
              sh.rej_t[k] = mt;
              sh.rej_d[k] = md;
            }
          }
          if (!acc) sh.n_k[k] = j;
        }
        const unsigned am = __ballot_sync(0xffffffffu, acc);
        const unsigned bm = __ballot_sync(0xffffffffu, bad);
        const unsigned im = __ballot_sync(0xffffffffu, inv);
        // helpers: the next position's rows already published for this
        // CTA's slice (each lane reads its candidate's record after its flag)
        unsigned hmask = 0;
        if (help) {
          const int hm = sh.hseen;
          const int jn = j + 1;
          if (hm && jn < gamma && am && !im) {
            bool ready = false;
            if (k < K && (am >> k & 1u)) {
              const size_t rec = hrec(b, jn, 1 + k);
              if (ld_acquire_gpu(p.hflag + rec)) {
                const float2 v = __ldcg(p.hpart + rec);
                sh.hv[1 + k] = MS{v.x, v.y};
                ready = true;
              }
            }
            hmask = __ballot_sync(0xffffffffu, ready) << 1;
            if (lane == 0) {
              const size_t rec = hrec(b, jn, 0);
              if (ld_acquire_gpu(p.hflag + rec)) {
                const float2 v = __ldcg(p.hpart + rec);
                sh.hv[0] = MS{v.x, v.y};
                hmask |= 1u;
              }
            }
          }
          if (lane == 0) {  // publish progress; take the next position
            atomicMax(p.hpos + (size_t)b * kHelpRanks + rank, (j + 2) * (K + 1));
            if (rank == 0) {
              st_relaxed_gpu(p.oalive + b, (int)am);
              st_relaxed_gpu(p.opos + b, j + 1);
            }
          }
        }
        __syncwarp();  // the lanes' n_k / rejection stats are visible
        if (lane == 0) {
          sh.alive = am;
          if (bm) sh.bad_token = 1;
          if (im) sh.invalid = 1;
          KSched &sc = sh.sc;
          sc.skip = hmask;
          sc.decided = j + 1;
          sc.alive = am;
          if (!am || im || j == gamma - 1) fu.end_scan(sc, sh);
          fu.pump(sc, ps, consumed);
        }
      }
      __syncthreads();
      if (sh.invalid || !sh.alive) break;
    }
    // --------------------------- selection and final token ---------------
    const int ksel = sh.sc.ksel, nsel = sh.sc.nsel, fkind = sh.sc.fkind;
    const bool invalid = sh.invalid;
    int t = -1;
    float prob = 0.f;
    bool inv_final = false;
    int zero_mass = 0;
    bool writer = (rank == 0 && warp == 0);
    if (!invalid) {
      const bool bonus = fkind == 2;
      MS mt = sh.rej_t[ksel], md = sh.rej_d[ksel];
      int gt = GREEDY && !bonus ? sh.rej_am[ksel] : -1;
      if (bonus) {  // the target row gamma of the selection
        stream_row(0);
        exchange(1, seqpar);
        if constexpr (GREEDY) {
          const AM a = sh.amrg[0];
          inv_final = a.bad || !(a.v > -kInf);
          gt = a.i;
        } else {
          mt = sh.mrg[0];
          inv_final = !ms_valid(mt);
        }
        if (tid == 0) {
          sh.sc.bdone = inv_final ? 2 : 1;
          fu.pump(sh.sc, ps, consumed);
        }
        md = ms_empty();
      }
      if (!inv_final) {
        if constexpr (GREEDY) {
          t = gt;
          prob = 1.f;
        } else {
          const bool has_q = !bonus;
          Weight W;
          W.k2 = k2;
          W.mtk = mt.m * k2;
          W.ist = 1.f / mt.s;
          W.mdk = md.m * k2;
          W.cq = 1.f / md.s;
          const float u = p.uniforms[((size_t)b * K + ksel) * G1 + gamma];
          // the draw's pair (or the bonus row) streams through the ring
          // again in two-row stages; the segment masses land in segmass
          cluster_total(cluster, sh.draw, segmass, sl, u, par, [&] {
            for (int c = 0; c < nchd; ++c) {
              const int cn = min(kStg, nv - c * kStg);
              consume([&](const uint4 *A) {
                const uint4 *Bq = A + kStg;
                for (int g = warp; g * 32 < cn; g += kWarps) {
                  const int i = g * 32 + lane;
                  float acc = 0.f;
                  if (i < cn) {
                    float w[VW];
                    weights<DT, VW>(sget<DT, VW>(A, i),
                                    sget<DT, VW>(has_q ? Bq : A, i), has_q,
                                    W, w);
#pragma unroll
                    for (int e = 0; e < VW; ++e) acc += w[e];
                  }
                  acc = warp_down_sum(acc);
                  if (lane == 0) segmass[c * (kStg / 32) + g] = acc;
                }
              });
            }
          });
          const char *trow = fu.trow(b, ksel, nsel);
          const GR ra{trow};
          const GR rb{has_q ? fu.drow(b, nsel) : trow};
          DrawOut o = draw_pick<DT, VW>(cluster, sh.draw, segmass, ra, rb,
                                        has_q, W, sl);
          if (o.owner < 0) {  // zero residual mass: draw from p instead
            zero_mass = 1;
            __syncthreads();
            o = kr_redraw<DT, VW>(cluster, sh, segmass, sl, trow, W, u, par);
          }
          writer = (o.owner == rank && warp == 0);
          t = o.t;
          prob = (float)((double)o.wt / o.N);
        }
      }
    }
    const bool bad_seq = invalid || inv_final;
    if (writer) {
      for (int i = lane; i <= gamma; i += 32) {
        int v = -1;
        if (!bad_seq) {
          if (i < nsel) v = p.tokens[((size_t)b * K + ksel) * gamma + i];
          else if (i == nsel) v = t;
        }
        p.out_tokens[(size_t)b * G1 + i] = v;
      }
      if (p.n_per_cand)
        for (int k = lane; k < K; k += 32)
          p.n_per_cand[(size_t)b * K + k] = bad_seq ? -1 : sh.n_k[k];
      if (lane == 0) {
        p.n_acc[b] = bad_seq ? -1 : nsel;
        p.sel_k[b] = bad_seq ? -1 : ksel;
        if (p.out_prob) p.out_prob[b] = bad_seq ? 0.f : prob;
        status_or(p.dev_status, (sh.bad_token ? SD_DEV_BAD_TOKEN : 0) |
                                    (bad_seq ? SD_DEV_NONFINITE : 0) |
                                    (zero_mass ? SD_DEV_ZERO_MASS : 0));
      }
    }
    if (help && tid == 0)  // no more helpers for this sequence
      atomicMax(p.hpos + (size_t)b * kHelpRanks + rank, gamma * (K + 1));
    __syncthreads();
    b = sh.sc.next;  // learnt at this sequence's first exchange
    seqpar ^= 1;
    __syncthreads();  // every thread has read it before thread 0 resets it
    if (tid == 0) {
      KSched &sc = sh.sc;
      sc.dseq = b;
      sc.decided = 0;
      sc.alive = full;
      sc.done = 0;
      sc.fkind = 0;
      sc.bdone = 0;
      sc.next = -1;
      fu.pump(sc, ps, consumed);
    }
    __syncthreads();
  }
  if (help) {
    // Nothing left to verify (the ring is idle: everything issued was
    // consumed): compute this CTA's slice of the rows of positions ahead of
    // the scans still running, nearest to its owner's position first.
    if (tid == 0) {
      if (rank == 0) st_relaxed_gpu(p.active + cid, 0);
      st_relaxed_gpu(p.helping, 1);
    }
    for (int round = 0; round < gamma * (K + 1) * p.B; ++round) {
      if (warp == 0) {
        int bs = -1, bpri = 0x7fffffff;
        for (int c = lane; c < p.nclusters; c += 32) {
          const int a = ld_relaxed_gpu(p.active + c);
          if (a <= 0) continue;
          const int s = a - 1;
          const int h =
              ld_relaxed_gpu(p.hpos + (size_t)s * kHelpRanks + rank) / (K + 1);
          if (h >= gamma) continue;
          const int pri = h - ld_relaxed_gpu(p.opos + s);
          if (pri < bpri) {
            bpri = pri;
            bs = s;
          }
        }
        for (int o = 16; o; o >>= 1) {  // lowest priority, then lowest s
          const int op = __shfl_xor_sync(0xffffffffu, bpri, o);
          const int os = __shfl_xor_sync(0xffffffffu, bs, o);
          if (op < bpri || (op == bpri && (unsigned)os < (unsigned)bs)) {
            bpri = op;
            bs = os;
          }
        }
        if (lane == 0) {
          int jc = gamma, rc = 0;
          if (bs >= 0) {  // one row; position 0 and dead candidates skipped
            int *hp = p.hpos + (size_t)bs * kHelpRanks + rank;
            const unsigned al = (unsigned)ld_relaxed_gpu(p.oalive + bs);
            for (int t = 0; t < 2 * (K + 1); ++t) {
              const int idx = atomicAdd(hp, 1);
              jc = idx / (K + 1);
              rc = idx % (K + 1);
              if (jc >= gamma) break;
              if (jc > 0 && (rc == 0 || (al >> (rc - 1) & 1u))) break;
            }
          }
          sh.hs = bs;
          sh.hj = jc;
          sh.hr = rc;
        }
      }
      __syncthreads();
      const int hs = sh.hs, hj = sh.hj, hr = sh.hr;
      if (hs < 0) break;
      if (hj > 0 && hj < gamma) {
        {
          const int row = hr;  // 0: the draft row; 1 + k: candidate k's
          if (tid == 0) {  // the row as the producer's current item
            const char *src = row == 0 ? fu.drow(hs, hj) : fu.trow(hs, row - 1, hj);
            ps.pa = src + (size_t)sl.vbeg * 16;
            ps.pb = nullptr;
            ps.prem = nv;
            ps.pstg = kStageVecs;
            fu.pump(sh.sc, ps, consumed);
          }
          stream_row(0);
          __syncthreads();
          if (tid == 0) {  // folded as the owner's exchange folds
            MS a = sh.wpart[0][0];
            for (int w = 1; w < kWarps; ++w) a = ms_merge(a, sh.wpart[0][w], k2);
            const size_t rec = hrec(hs, hj, row);
            __stcg(p.hpart + rec, make_float2(a.m, a.s));
            st_release_gpu(p.hflag + rec, 1);
          }
          __syncthreads();
        }
      }
      __syncthreads();
    }
  }
  cluster.sync();  // no CTA leaves while a peer may still read its smem
}

using KRKernel = void (*)(const KRParams);

static KRKernel pick_kr(int dt, bool greedy) {
  if (dt == SD_F32)
    return greedy ? kcand_ring_kernel<0, 4, true> : kcand_ring_kernel<0, 4, false>;
  return greedy ? kcand_ring_kernel<1, 8, true> : kcand_ring_kernel<1, 8, false>;
}

// Workspace layout: the work counter (byte 0) and the helping flag (byte 4),
// then the helping records; everything before the partials is cleared on
// the stream before each launch.
struct KHelpLayout {
  size_t active, opos, oalive, hpos, hflag, hpart, zero_end, total;
};
constexpr int kKHelpMaxClusters = 1024;
constexpr size_t kKHelpMaxWs = (size_t)64 << 20;

static KHelpLayout kh_layout(int B, int K, int gamma) {
  auto r256 = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t nb = B > 0 ? (size_t)B : 0;
  const size_t recs = nb * (size_t)(gamma > 0 ? gamma : 0) * (size_t)(K + 1) *
                      kHelpRanks;
  KHelpLayout L;
  L.active = 256;
  L.opos = L.active + r256((size_t)kKHelpMaxClusters * 4);
  L.oalive = L.opos + r256(nb * 4);
  L.hpos = L.oalive + r256(nb * 4);
  L.hflag = L.hpos + r256(nb * kHelpRanks * 4);
  L.hpart = L.hflag + r256(recs * 4);
  L.zero_end = L.hpart;
  L.total = L.hpart + recs * 8;
  return L;
}

// Bytes the helping records need (0: K of 32, or too large; the call then
// runs without helping).
size_t kcand_help_workspace(int B, int K, int gamma) {
  if (B <= 0 || K < 1 || K > 31 || gamma < 1) return 0;
  const size_t t = kh_layout(B, K, gamma).total;
  return t <= kKHelpMaxWs ? t : 0;
}

// Launch for 16-byte aligned rows.  *launched = false (and SD_OK) when the
// shapes do not suit the streaming kernel.
sd_status kcand_ring_launch(const void *target, const void *draft,
                            sd_dtype dt, const int32_t *tokens,
                            const float *uniforms, int B, int K, int gamma,
                            int V, float T, int32_t *n_acc, int32_t *sel_k,
                            int32_t *out_tokens, int32_t *n_per_cand,
                            float *out_prob, int32_t *dev_status, void *ws,
                            size_t ws_bytes, cudaStream_t stream,
                            bool *launched) {
  *launched = false;
  if (tune(SD_TUNE_KCAND_RING) == 0) return SD_OK;
  const bool greedy = (T == 0.f);
  const int vw = dt == SD_F32 ? 4 : 8;
  const long long nvec = V / vw;
  KRKernel kern = pick_kr(dt, greedy);
  auto smem_for = [&](int cl) {
    const long long per_cta = (nvec + cl - 1) / cl;
    const size_t seg = ((size_t)((per_cta + 31) / 32) * 4 + 127) / 128 * 128;
    return seg + (size_t)kRingBytes;
  };
  // the largest cluster at which all B sequences are resident at once (at
  // least one full stage per slice), else single CTAs and the work counter
  int CL = 1, maxc = 0;
  const int forced = tune(SD_TUNE_CLUSTER);
  for (int c = 16; c >= 1; c /= 2) {
    if (forced && c != forced && c != 1) continue;
    if (c > 1 && nvec / c < kStageVecs && !forced) continue;
    int mc = 0;
    sd_status st = max_active_clusters((const void *)kern, c, smem_for(c), &mc);
    if (st != SD_OK) return st;
    if (B <= mc || c == 1 || forced) {
      CL = c;
      maxc = mc;
      break;
    }
  }
  const size_t smem = smem_for(CL);
  if (smem > 64 * 1024 || maxc <= 0) return SD_OK;
  if (!ws || ws_bytes < 256)
    return fail(SD_ERR_INVALID_ARG, "workspace of >= 256 bytes required");
  KRParams prm;
  prm.target = target;
  prm.draft = draft;
  prm.tokens = tokens;
  prm.uniforms = uniforms;
  prm.B = B;
  prm.K = K;
  prm.gamma = gamma;
  prm.V = V;
  prm.k2 = greedy ? 0.f : (float)(1.4426950408889634 / (double)T);
  prm.n_acc = n_acc;
  prm.sel_k = sel_k;
  prm.out_tokens = out_tokens;
  prm.n_per_cand = n_per_cand;
  prm.out_prob = out_prob;
  prm.dev_status = dev_status;
  prm.queue = static_cast<int *>(ws);
  prm.nclusters = B < maxc ? B : maxc;
  prm.seg_bytes = (int)(smem - kRingBytes);
  prm.helping = prm.active = prm.opos = prm.oalive = prm.hpos = nullptr;
  prm.hflag = nullptr;
  prm.hpart = nullptr;
  const size_t hws = kcand_help_workspace(B, K, gamma);
  if (!greedy && tune(SD_TUNE_HELPERS) != 0 && hws != 0 && ws_bytes >= hws &&
      CL <= kHelpRanks && prm.nclusters <= kKHelpMaxClusters) {
    const KHelpLayout L = kh_layout(B, K, gamma);
    char *w = static_cast<char *>(ws);
    prm.helping = reinterpret_cast<int *>(w + 4);
    prm.active = reinterpret_cast<int *>(w + L.active);
    prm.opos = reinterpret_cast<int *>(w + L.opos);
    prm.oalive = reinterpret_cast<int *>(w + L.oalive);
    prm.hpos = reinterpret_cast<int *>(w + L.hpos);
    prm.hflag = reinterpret_cast<int *>(w + L.hflag);
    prm.hpart = reinterpret_cast<float2 *>(w + L.hpart);
    SDV_CUDA(cudaMemsetAsync(ws, 0, L.zero_end, stream));
  } else {
    SDV_CUDA(cudaMemsetAsync(ws, 0, sizeof(int), stream));
  }
  void *args[] = {&prm};
  *launched = true;
  return launch_clusters((const void *)kern, prm.nclusters, CL, smem, stream,
                         args);
}

}  // namespace sdv
