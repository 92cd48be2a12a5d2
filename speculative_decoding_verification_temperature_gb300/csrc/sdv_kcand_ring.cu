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
};

constexpr int kKRows = SD_MAX_K + 1;  // draft row + one per candidate

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
        if (!GREEDY) ra = drow(b, j);
      } else if (sc.pkind == 1) {  // target rows of the live candidates
        const unsigned alive = j == 0 ? full() : sc.alive;
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

  if (tid == 0) fu.pump(sh.sc, ps, consumed);
  while (b < p.B) {
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
      int r = 0;
      if (!GREEDY) stream_row(r++);
      for (int k = 0; k < K; ++k)
        if (alive >> k & 1u) stream_row(r++);
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
        __syncwarp();  // the lanes' n_k / rejection stats are visible
        if (lane == 0) {
          sh.alive = am;
          if (bm) sh.bad_token = 1;
          if (im) sh.invalid = 1;
          KSched &sc = sh.sc;
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
  cluster.sync();  // no CTA leaves while a peer may still read its smem
}

using KRKernel = void (*)(const KRParams);

static KRKernel pick_kr(int dt, bool greedy) {
  if (dt == SD_F32)
    return greedy ? kcand_ring_kernel<0, 4, true> : kcand_ring_kernel<0, 4, false>;
  return greedy ? kcand_ring_kernel<1, 8, true> : kcand_ring_kernel<1, 8, false>;
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
  SDV_CUDA(cudaMemsetAsync(ws, 0, sizeof(int), stream));
  void *args[] = {&prm};
  *launched = true;
  return launch_clusters((const void *)kern, prm.nclusters, CL, smem, stream,
                         args);
}

}  // namespace sdv
