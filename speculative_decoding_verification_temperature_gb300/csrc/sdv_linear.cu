// sdv_linear.cu -- linear verify ("01 · Draft-then-verify", Algorithm 1 and
// the spec_step listing of section 4) as one persistent kernel.
//
// Design.  One thread-block cluster verifies one sequence at a time; the
// vocabulary axis of every row is cut into one slice per CTA of the
// cluster.  Positions are scanned left to right: at position i each CTA
// streams its slice of target row i and draft row i once (16-byte loads,
// single-pass online max / sum of 2^(z log2e / T)), the CTAs exchange their
// partial (max, sum) pairs through distributed shared memory, and every CTA
// merges them in rank order, so all CTAs reach the same accept decision
// r_i <= p_i(x_i) / q_i(x_i) without another barrier.  The scan stops at the
// first rejection: rows after it are never read.  The correction
// norm(max(0, p_n - q_n)) (section 2.1) or the bonus p_gamma is then drawn by
// inverse CDF over the same slices: a second pass (from L2: the rows were
// just read) writes per-segment masses, the cluster agrees on the slice
// holding u * N, and one warp scans one 32-vector segment.
//
// Clusters take sequences from a work counter, so short and long scans
// balance across the GPU.  Greedy (T == 0) compares draft ids with the
// row argmax (section 2.2) and reads no draft logits.  Once the counter is
// exhausted, clusters left without a sequence help the scans still running
// (LinearParams: helping).  The FAN instantiation is the verify fused with
// the Saguaro fan-out (sd_verify_linear_fanout): CTAs left without a
// sequence compute the fan-out's top-F rows, settling the rows the scans
// streamed from records the scans keep (LinearParams: fused fan-out).
//
// Two ways to read a step's slices: through a ring of shared-memory stages
// filled by TMA bulk copies (cp.async.bulk, one mbarrier per stage), used
// when rows are 16-byte aligned; or 16-byte loads from global memory with
// several in flight per thread.  The draw streams the last step's slices
// again (they were just read: from L2).
#include <type_traits>

#include "sdv_device.cuh"
#include "sdv_fanrow.cuh"
#include "sdv_host.cuh"
#include "sdv_ring.cuh"
#include "sdv_tma.cuh"

#ifndef SDV_LDG_MINB
#define SDV_LDG_MINB 2
#endif

namespace sdv {

struct LinearParams {
  const void *target;  // [B, gamma+1, V]
  const void *draft;   // [B, d_seq_rows, V]
  const int32_t *tokens;
  const float *uniforms;
  int B, gamma, V;
  long long d_seq_rows;  // rows per sequence in the draft tensor
  float k2;              // log2(e) / T
  int32_t *n_acc;
  int32_t *out_tokens;
  float *out_prob;
  float *out_accept;
  float *out_resid;
  int32_t *dev_status;
  int *queue;  // nullable: then cluster c verifies sequence c only
  int nclusters;
  int seg_bytes;   // bytes of the segment-mass array (multiple of 128)
  int slice_vecs;  // capacity of each slice buffer in 16-byte vectors (TMA)
  int spec;        // let a cluster's last sequence read ahead (0: never)
  // Helping (all null when off).  Once the work counter is exhausted, a
  // cluster with nothing left to verify computes row statistics for the
  // sequences other clusters are still scanning: each of its CTAs takes a
  // position ahead of a running scan, computes its own slice's partial of
  // that position's rows (the same code and slice as the owner's CTA of the
  // same rank, hence the same bits), stores it and raises a flag.  An owner
  // CTA that finds the flag of its slice raised copies the partial instead
  // of streaming the slice.  Nobody ever waits on a flag.
  int *helping;     // set once a cluster has started helping
  int *active;      // [nclusters]: sequence + 1 being verified, or 0
  int *opos;        // [B]: the owner's current position
  int *hpos;        // [B][kHelpRanks]: next position to hand to a helper
  int *hflag;       // [B][gamma+1][kHelpRanks]: partial published
  uint4 *hpart;     // [B][gamma+1][kHelpRanks]: the partials
  // Fused fan-out (the FAN kernels; sd_verify_linear_fanout).  Draft row j
  // of every sequence (j = 0..gamma, the draft tensor holding gamma + 1
  // rows) gets its exact top-fF[j] keys.  While a scan streams draft row j
  // each of its threads also keeps its best vector (sdv_fanrow.cuh) and
  // stores it; fcov[b] then says that rows 0..fcov[b]-1 of sequence b have
  // their records.  A CTA with no sequence left to verify takes rows from
  // the row counter, one CTA per row, the sequences handed out last first:
  // a covered row from its records when they determine the top-F, any other
  // row whole.
  int32_t *fan_tokens;  // [B, ftotal]
  float *fan_logit;     // nullable
  int fF[SD_MAX_K + 1], foff[SD_MAX_K + 1];
  int ftotal;
  int *fq;        // the row counter
  int *fcov;      // [B] (null: no records kept)
  uint4 *cand_v;  // [B][gamma][CL][kThreads]: each thread's best vector
  int *cand_i;    // its index in the row
  float *cand_t;  // the thread's largest other vector maximum
};

constexpr int kHelpRanks = 16;  // record stride: the largest cluster

constexpr int kMaxW = 4;  // positions per step when a cluster speculates


struct StepResult {
  int kind;   // 0 continue, 1 reject at n, 2 bonus, 3 unusable row
  int n;      // accepted drafts so far
  int tok;    // greedy: argmax of the final row
  int bad;    // a bad token was seen
  MS mt, md;  // merged stats of the final rows
};

struct LinearSmem {
  MS red[2][kWarps];
  AM ared[kWarps];
  // [parity][row]: this CTA's partials of the step's rows (peers read)
  union {
    MS part[2][2 * kMaxW];
    AM apart[2][kMaxW];
  };
  MS mrg[2 * kMaxW];      // merged stats of this step's rows
  AM amrg[kMaxW];
  int next_seq[2];
  // helping: flags of this step's positions, consecutive published
  // positions after the step (this CTA's slice; peers read it), the
  // cluster's minimum of those, a helper's assignment
  int hready[kMaxW];
  uint4 hv[kMaxW];  // the published partials of this step's positions
  int rcnt[2];
  int wready;
  int hseen[2];  // rank 0: the helping flag as read at the step's start
  int hnext;     // rank 0's, read by every CTA after the step's barrier
  int hs, hj;
  // gathered for the accept tests of this step's positions
  int gx[kMaxW];
  float gzt[kMaxW], gzd[kMaxW], gr[kMaxW];
  StepResult res;
  DrawSmem draw;
};

// The FAN kernels' shared memory: a row's top-F and the filters' state.
struct LinearSmemFan : LinearSmem {
  uint64_t fout[SD_MAX_FANOUT];
  uint32_t fth;    // the warp filters' CTA threshold
  uint32_t t2max;  // ord32 of the largest t2 of a row's records
  int fitem, fcov;
};

template <int DT, int VW, bool GREEDY, bool RING, bool FAN = false>
__global__ void __launch_bounds__(kThreads, RING ? 4 : 2)
    linear_verify_kernel(const LinearParams p) {
  static_assert(RING || !FAN, "the fused fan-out needs the ring");
  using SMT = std::conditional_t<FAN, LinearSmemFan, LinearSmem>;
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ SMT sh;
  __shared__ uint64_t bars[2 * kStages];
  using GR = GRow<DT, VW>;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int CL = (int)cluster.num_blocks();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = p.V, gamma = p.gamma;
  const Slice sl = make_slice(V / VW, rank, CL);
  const size_t rowb = (size_t)V * elt_bytes<DT>();
  const char *tbase = static_cast<const char *>(p.target);
  const char *dbase = static_cast<const char *>(p.draft);
  const float k2 = p.k2;
  // dynamic shared memory: segment masses, then the ring stages
  float *segmass = reinterpret_cast<float *>(dsm);
  Ring rg;
  rg.buf = reinterpret_cast<uint4 *>(dsm + p.seg_bytes);
  rg.full = bars;
  rg.empty = bars + kStages;
  rg.dev_status = p.dev_status;
  if constexpr (FAN) {
    if (tid == 0) {
      sh.fth = 0;
      sh.t2max = 0;
    }
  }
  if (RING) ring_init(rg);  // (a block barrier)
  auto trow_of = [&](int s, int j) {
    return tbase + ((size_t)s * (gamma + 1) + j) * rowb;
  };
  auto drow_of = [&](int s, int j) {
    return dbase + ((size_t)s * p.d_seq_rows + j) * rowb;
  };
  // this CTA's partial of position j of sequence s, valid at thread 0:
  // (max, sum) of the target and the draft row, or the target's argmax
  auto slice_stats = [&](int s, int j) -> uint4 {
    const char *trow = trow_of(s, j);
    if constexpr (GREEDY) {
      AM a = am_empty();
      if constexpr (RING) ring_argmax<DT, VW>(rg, trow, sl, a);
      else argmax_pass<DT, VW>(GR{trow}, sl, a);
      a = block_reduce_am(a, sh.ared);
      return make_uint4(__float_as_uint(a.v), (unsigned)a.i, (unsigned)a.bad,
                        0u);
    } else {
      const bool has_d = j < gamma;
      const char *drow = has_d ? drow_of(s, j) : nullptr;
      MS st[2] = {ms_empty(), ms_empty()};
      if constexpr (RING) {
        ring_stats<DT, VW>(rg, trow, drow, sl, k2, st[0], st[1]);
      } else {
        stats_pass<DT, VW>(GR{trow}, GR{drow}, has_d, sl, k2, st[0], st[1]);
      }
      block_reduce_ms<2>(st, k2, sh.red);
      return make_uint4(__float_as_uint(st[0].m), __float_as_uint(st[0].s),
                        __float_as_uint(st[1].m), __float_as_uint(st[1].s));
    }
  };
  // FAN: the stats of position j while this CTA's threads also keep their
  // best vectors of its draft row and store them (same arithmetic as
  // slice_stats)
  auto cand_stats = [&](int s, int j) -> uint4 {
    if constexpr (FAN && !GREEDY) {
      const char *trow = trow_of(s, j), *drow = drow_of(s, j);
      MS st[2] = {ms_empty(), ms_empty()};
      VecTop<DT, VW> T;
      vec_top_init(T);
      ring_pass(rg, trow, drow, sl, [&](const uint4 *A, const uint4 *Bp,
                                        int v0, int n) {
        for (int i = tid; i < n; i += kThreads) {
          ms_add<DT, VW>(st[0], sget<DT, VW>(A, i), k2);
          const Raw<DT, VW> d = sget<DT, VW>(Bp, i);
          float vm;
          ms_add_v<DT, VW>(st[1], d, k2, vm);
          vec_top_add(T, d, vm, v0 + i);
        }
      });
      const size_t r = ((size_t)s * gamma + j) * CL * kThreads +
                       (size_t)rank * kThreads + tid;
      // a NaN or an infinity among this thread's elements leaves its sum
      // non-finite (the row is then read whole)
      vec_top_store(T, isfinite(st[1].s), p.cand_v + r, p.cand_i + r,
                    p.cand_t + r);
      block_reduce_ms<2>(st, k2, sh.red);
      return make_uint4(__float_as_uint(st[0].m), __float_as_uint(st[0].s),
                        __float_as_uint(st[1].m), __float_as_uint(st[1].s));
    } else {
      return slice_stats(s, j);
    }
  };
  const bool help = p.hflag != nullptr;
  const int cid = (int)(blockIdx.x / CL);
  auto hrec = [&](int s, int j) {  // index of this CTA's record
    return ((size_t)s * (gamma + 1) + j) * kHelpRanks + rank;
  };
  bool hmode = false;  // helpers are running: look for their partials

  int par = 0, seqpar = 0;
  int seq = (int)(blockIdx.x / CL);
  while (seq < p.B) {
    if (rank == 0 && tid == 0) {
      sh.next_seq[seqpar] =
          p.queue ? p.nclusters + atomicAdd(p.queue, 1) : p.B;
      if (help) st_relaxed_gpu(p.active + cid, seq + 1);
    }
    // ---------------- scan: positions [i, i + w) per step -----------------
    // w stays 1 while the work counter still hands out sequences; once this
    // cluster holds its last sequence (nothing else to overlap with), w
    // doubles each step: later positions are read speculatively, which
    // shortens the longest scans at the end of the call.
    int i = 0, w = 1;
    bool last_seq = false, first = true;
    StepResult R;
    for (;;) {
      const int jend = min(i + w, gamma + 1);
      const int np = jend - i;
      // gathers for the accept tests (used after the merge), by warp 1:
      // thread 0 goes straight on to issue the step's copies
      if (tid >= 32 && tid < 32 + np) {
        const int j = i + tid - 32;
        int x = -1;
        float zt = 0.f, zd = 0.f, r = 0.f;
        if (j < gamma) {
          x = p.tokens[(size_t)seq * gamma + j];
          if (!GREEDY && x >= 0 && x < V) {
            zt = load_logit<DT>(trow_of(seq, j), x);
            zd = load_logit<DT>(drow_of(seq, j), x);
          }
          if (!GREEDY) r = p.uniforms[(size_t)seq * (gamma + 1) + j];
        }
        sh.gx[tid - 32] = x;
        sh.gzt[tid - 32] = zt;
        sh.gzd[tid - 32] = zd;
        sh.gr[tid - 32] = r;
      }
      if (help) {
        if (tid == 63 && rank == 0) sh.hseen[par] = ld_relaxed_gpu(p.helping);
        if (tid == 0) {  // the owner computes [i, jend) unless published
          atomicMax(p.hpos + (size_t)seq * kHelpRanks + rank, jend);
          if (rank == 0) st_relaxed_gpu(p.opos + seq, i);
        }
        if (hmode) {
          if (tid < np) {  // each lane reads its record after its flag
            const size_t rec = hrec(seq, i + tid);
            const int f = ld_acquire_gpu(p.hflag + rec);
            sh.hready[tid] = f;
            if (f) sh.hv[tid] = __ldcg(p.hpart + rec);
          }
          __syncthreads();
        }
      }
      if (RING && last_seq && p.spec >= 2 && tid == 0) {
        // the GPU is emptying out: ask for this step's and the next step's
        // rows at once (into L2), so the ring below streams from L2
        const uint32_t sb = (uint32_t)(sl.vend - sl.vbeg) * 16u;
        const int jpre = min(i + 3 * w, gamma + 1);
        for (int j = i; j < jpre && sb; ++j) {
          prefetch_l2(trow_of(seq, j) + (size_t)sl.vbeg * 16, sb);
          if (!GREEDY && j < gamma)
            prefetch_l2(drow_of(seq, j) + (size_t)sl.vbeg * 16, sb);
        }
      }
      for (int t = 0; t < np; ++t) {
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (hmode && sh.hready[t]) {
          v = sh.hv[t];
        } else if (FAN && !GREEDY && p.fcov && i + t < gamma &&
                   p.fF[i + t] > 0) {
          v = cand_stats(seq, i + t);
        } else {
          v = slice_stats(seq, i + t);
        }
        if (tid == 0) {
          if constexpr (GREEDY) {
            sh.apart[par][t] = AM{__uint_as_float(v.x), (int)v.y, (int)v.z};
          } else {
            sh.part[par][2 * t] = MS{__uint_as_float(v.x), __uint_as_float(v.y)};
            sh.part[par][2 * t + 1] =
                MS{__uint_as_float(v.z), __uint_as_float(v.w)};
          }
        }
        __syncthreads();
      }
      if (hmode && warp == 0) {  // published positions right after the step
        const int j = jend + lane;
        const bool ok = lane < kMaxW && j <= gamma &&
                        ld_acquire_gpu(p.hflag + hrec(seq, j)) != 0;
        const unsigned m = __ballot_sync(0xffffffffu, ok);
        if (lane == 0) sh.rcnt[par] = __ffs(~m) - 1;
      }
      const int nrows = GREEDY ? np : 2 * np;
      cluster.sync();
      // every CTA merges the CL partials of every row in the same order
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
      if (hmode && warp == kWarps - 1) {
        int c = kMaxW;
        if (lane < CL) c = cluster.map_shared_rank(&sh, lane)->rcnt[par];
        for (int o = 16; o; o >>= 1) c = min(c, __shfl_xor_sync(0xffffffffu, c, o));
        if (lane == 0) sh.wready = c;
      }
      // every CTA takes rank 0's reading, so the whole cluster switches to
      // looking for published partials at the same step
      if (help && !hmode && tid == kThreads - 32)
        sh.hnext = cluster.map_shared_rank(&sh, 0)->hseen[par];
      __syncthreads();
      par ^= 1;
      if (tid == 0) {  // the accept tests of this step, in position order
        StepResult q = (i == 0) ? StepResult{0, 0, -1, 0, ms_empty(), ms_empty()} : sh.res;
        q.kind = 0;
        for (int t = 0; t < np && !q.kind; ++t) {
          const int j = i + t;
          const int x = sh.gx[t];
          const bool bad = j < gamma && (x < 0 || x >= V);
          q.bad |= bad;
          bool invalid, acc = false;
          float accp = 0.f;
          if constexpr (GREEDY) {
            const AM a = sh.amrg[t];
            invalid = a.bad || !(a.v > -kInf);
            acc = !invalid && j < gamma && x == a.i;
            accp = acc ? 1.f : 0.f;
            q.tok = a.i;
          } else {
            const MS mt = sh.mrg[2 * t], md = sh.mrg[2 * t + 1];
            invalid = !ms_valid(mt) || (j < gamma && !ms_valid(md));
            if (!invalid && j < gamma && !bad) {
              const float rho =
                  accept_ratio(sh.gzt[t], sh.gzd[t], mt, md, k2);
              acc = sh.gr[t] <= rho;
              accp = fminf(1.f, rho);
            }
            q.mt = mt;
            q.md = md;
          }
          if (rank == 0 && p.out_accept && j < gamma && !invalid)
            p.out_accept[(size_t)seq * gamma + j] = accp;
          if (invalid) q.kind = 3;
          else if (j == gamma) q.kind = 2;
          else if (!acc) q.kind = 1;
          else ++q.n;
        }
        sh.res = q;
      }
      __syncthreads();
      R = sh.res;
      if constexpr (FAN && !GREEDY) {
        // every CTA stored the records of [i, jend) before the barrier
        if (p.fcov && rank == 0 && tid == 0)
          st_release_gpu(p.fcov + seq, min(jend, gamma));
      }
      if (R.kind) break;
      i = jend;
      if (first) {  // after the first step: is this the cluster's last?
        last_seq = cluster.map_shared_rank(&sh, 0)->next_seq[seqpar] >= p.B;
        first = false;
      }
      w = (last_seq && p.spec) ? min(2 * w, kMaxW) : 1;
      if (hmode) w = max(w, sh.wready);
      if (help && !hmode) hmode = sh.hnext != 0;
    }
    const int n = R.n, kind = R.kind, bad_token = R.bad;

    if (kind == 3) {  // unusable row: outputs -1
      if (rank == 0) {
        for (int t = tid; t <= gamma; t += kThreads)
          p.out_tokens[(size_t)seq * (gamma + 1) + t] = -1;
        if (p.out_accept)
          for (int t = n + tid; t < gamma; t += kThreads)
            p.out_accept[(size_t)seq * gamma + t] = -1.f;
        if (tid == 0) {
          p.n_acc[seq] = -1;
          if (p.out_prob) p.out_prob[seq] = 0.f;
          status_or(p.dev_status,
                    SD_DEV_NONFINITE | (bad_token ? SD_DEV_BAD_TOKEN : 0));
        }
      }
    } else if (GREEDY) {
      if (rank == 0) {
        for (int t = tid; t <= gamma; t += kThreads) {
          int v = -1;
          if (t < n) v = p.tokens[(size_t)seq * gamma + t];
          else if (t == n) v = R.tok;
          p.out_tokens[(size_t)seq * (gamma + 1) + t] = v;
        }
        if (p.out_accept)
          for (int t = n + 1 + tid; t < gamma; t += kThreads)
            p.out_accept[(size_t)seq * gamma + t] = -1.f;
        if (tid == 0) {
          p.n_acc[seq] = n;
          if (p.out_prob) p.out_prob[seq] = 1.f;
          status_or(p.dev_status, bad_token ? SD_DEV_BAD_TOKEN : 0);
        }
      }
      if (p.out_resid) {
        float *res = p.out_resid + (size_t)seq * V;
        for (int j = sl.vbeg * VW + tid; j < sl.vend * VW; j += kThreads)
          res[j] = (j == R.tok) ? 1.f : 0.f;
      }
    } else {
      // correction (kind 1) or bonus (kind 2) by inverse CDF over the rows
      // of position n (streamed again: they were just read, so from L2)
      const char *trow = trow_of(seq, n);
      const char *drow = kind == 1 ? drow_of(seq, n) : nullptr;
      const GR ra{trow}, rb{drow ? drow : trow};
      bool has_q = kind == 1;
      Weight W;
      W.k2 = k2;
      W.mtk = R.mt.m * k2;
      W.ist = 1.f / R.mt.s;
      W.mdk = R.md.m * k2;
      W.cq = 1.f / R.md.s;
      const float u = p.uniforms[(size_t)seq * (gamma + 1) + gamma];
      int zero_mass = 0;
      DrawOut o;
      for (int attempt = 0; attempt < 2; ++attempt) {
        cluster_total(cluster, sh.draw, segmass, sl, u, par, [&] {
          if constexpr (RING) {
            ring_mass<DT, VW>(rg, trow, drow, has_q, W, sl, segmass);
          } else {
            mass_pass<DT, VW>(ra, rb, has_q, W, sl, segmass);
          }
        });
        o = draw_pick<DT, VW>(cluster, sh.draw, segmass, ra, rb, has_q, W, sl);
        if (o.owner >= 0) break;
        zero_mass = 1;  // residual of zero mass: draw from p_n instead
        has_q = false;
        __syncthreads();
      }
      if (o.owner == rank && warp == 0) {
        for (int t = lane; t <= gamma; t += 32) {
          int v = -1;
          if (t < n) v = p.tokens[(size_t)seq * gamma + t];
          else if (t == n) v = o.t;
          p.out_tokens[(size_t)seq * (gamma + 1) + t] = v;
        }
        if (p.out_accept)
          for (int t = n + 1 + lane; t < gamma; t += 32)
            p.out_accept[(size_t)seq * gamma + t] = -1.f;
        if (lane == 0) {
          p.n_acc[seq] = n;
          if (p.out_prob) p.out_prob[seq] = (float)((double)o.wt / o.N);
          status_or(p.dev_status, (bad_token ? SD_DEV_BAD_TOKEN : 0) |
                                      (zero_mass ? SD_DEV_ZERO_MASS : 0));
        }
      }
      if (p.out_resid)
        write_resid<DT, VW>(p.out_resid + (size_t)seq * V, ra, rb, has_q, W,
                            sl, o.N);
    }
    if (help && tid == 0)  // no more helpers for this sequence
      atomicMax(p.hpos + (size_t)seq * kHelpRanks + rank, gamma + 1);
    // next sequence (rank 0 published it before this sequence's first sync)
    seq = cluster.map_shared_rank(&sh, 0)->next_seq[seqpar];
    seqpar ^= 1;
    __syncthreads();
  }
  if (help) {
    // Nothing left to verify: compute this CTA's slice of positions ahead
    // of the scans still running, nearest to its owner's position first.
    if (tid == 0) {
      if (rank == 0) st_relaxed_gpu(p.active + cid, 0);
      st_relaxed_gpu(p.helping, 1);
    }
    for (int round = 0; round < (gamma + 1) * p.B; ++round) {
      if (warp == 0) {  // candidates: the sequences clusters published
        int bs = -1, bpri = 0x7fffffff;
        for (int c = lane; c < p.nclusters; c += 32) {
          const int a = ld_relaxed_gpu(p.active + c);
          if (a <= 0) continue;
          const int s = a - 1;
          const int h = ld_relaxed_gpu(p.hpos + (size_t)s * kHelpRanks + rank);
          if (h > gamma) continue;
          const int pri = h - ld_relaxed_gpu(p.opos + s);
          if (pri < bpri) { bpri = pri; bs = s; }
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
          int j = gamma + 1;
          if (bs >= 0) {  // position 0 is always the owner's own
            int *hp = p.hpos + (size_t)bs * kHelpRanks + rank;
            j = atomicAdd(hp, 1);
            if (j == 0) j = atomicAdd(hp, 1);
          }
          sh.hs = bs;
          sh.hj = j;
        }
      }
      __syncthreads();
      const int s = sh.hs, j = sh.hj;
      if (s < 0) break;
      if (j <= gamma) {
        const uint4 v = slice_stats(s, j);
        if (tid == 0) {
          __stcg(p.hpart + hrec(s, j), v);
          st_release_gpu(p.hflag + hrec(s, j), 1);
        }
      }
      __syncthreads();
    }
  }
  if constexpr (FAN) {
    // the fan-out rows, one CTA per row: sequences from the last handed out
    // (whose draft rows the scans read most recently, possibly still in L2)
    // to the first, rows in order
    const int K1 = gamma + 1, nitems = K1 * p.B;
    uint64_t *scratch = reinterpret_cast<uint64_t *>(rg.buf);  // ring idle
    // each fan-out row is read once: keep it from pushing out the lines the
    // scans still running read again (their draws)
    rg.policy = l2_evict_first_policy();
    for (;;) {
      if (tid == 0) {
        const int q = atomicAdd(p.fq, 1);
        sh.fitem = q;
        sh.fcov = (q < nitems && p.fcov)
                      ? ld_acquire_gpu(p.fcov + (p.B - 1 - q / K1)) : 0;
      }
      __syncthreads();
      const int q = sh.fitem, cov = sh.fcov;
      __syncthreads();
      if (q >= nitems) break;
      const int s = p.B - 1 - q / K1, j = q % K1;
      if (p.fF[j] == 0) continue;
      const size_t o = (size_t)s * p.ftotal + p.foff[j];
      int32_t *otok = p.fan_tokens + o;
      float *olog = p.fan_logit ? p.fan_logit + o : nullptr;
      if constexpr (!GREEDY) {
        if (j < cov) {  // the scan kept this row's best vectors
          const size_t r0 = ((size_t)s * gamma + j) * CL * kThreads;
          if (cta_vec_topf<DT, VW>(p.cand_v + r0, p.cand_i + r0,
                                   p.cand_t + r0, CL * kThreads, &sh.fth,
                                   &sh.t2max, scratch, sh.fout, p.fF[j],
                                   otok, olog, p.dev_status))
            continue;
        }
      }
      cta_row_topf<DT, VW>(rg, &sh.fth, scratch, sh.fout, drow_of(s, j), V,
                           p.fF[j], otok, olog, p.dev_status);
    }
  }
  cluster.sync();  // no CTA leaves while a peer may still read its smem
}

// ------------------------------------------------------------------ host

using LinearKernel = void (*)(const LinearParams);

template <int DT, int VW, bool RING>
static LinearKernel pick_linear_t(bool greedy) {
  return greedy ? linear_verify_kernel<DT, VW, true, RING>
                : linear_verify_kernel<DT, VW, false, RING>;
}

static LinearKernel pick_linear_fan(int dt, bool greedy) {
  if (dt == SD_F32)
    return greedy ? linear_verify_kernel<0, 4, true, true, true>
                  : linear_verify_kernel<0, 4, false, true, true>;
  return greedy ? linear_verify_kernel<1, 8, true, true, true>
                : linear_verify_kernel<1, 8, false, true, true>;
}

static LinearKernel pick_linear(int dt, bool vec, bool ring, bool greedy) {
  if (dt == SD_F32) {
    if (!vec) return pick_linear_t<0, 1, false>(greedy);
    return ring ? pick_linear_t<0, 4, true>(greedy)
                : pick_linear_t<0, 4, false>(greedy);
  }
  if (!vec) return pick_linear_t<1, 1, false>(greedy);
  return ring ? pick_linear_t<1, 8, true>(greedy)
              : pick_linear_t<1, 8, false>(greedy);
}

size_t allrows_workspace(int B, int gamma, int V, sd_dtype dt);

// Workspace layout: the work counter (byte 0) and the helping flag (byte 4)
// in the first 256 bytes, then the helping records; everything before the
// partials is cleared on the stream before each launch.
struct HelpLayout {
  size_t active, opos, hpos, hflag, hpart, zero_end, total;
};
constexpr int kHelpMaxClusters = 1024;
constexpr size_t kHelpMaxWs = 768 << 10;

static HelpLayout help_layout(int B, int gamma) {
  auto r256 = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t recs = (size_t)B * (gamma + 1) * kHelpRanks;
  HelpLayout L;
  L.active = 256;
  L.opos = L.active + r256((size_t)kHelpMaxClusters * 4);
  L.hpos = L.opos + r256((size_t)B * 4);
  L.hflag = L.hpos + r256((size_t)B * kHelpRanks * 4);
  L.hpart = L.hflag + r256(recs * 4);
  L.zero_end = L.hpart;
  L.total = L.hpart + recs * 16;
  return L;
}

// Bytes the helping records need (0: too many sequences x positions; the
// call then runs without helping).
size_t help_workspace(int B, int gamma) {
  if (B <= 0 || gamma < 0) return 0;
  const size_t t = help_layout(B, gamma).total;
  return t <= kHelpMaxWs ? t : 0;
}

bool use_allrows(int B, int gamma, int V, sd_dtype dt, const void *target,
                 const void *draft, float T, const float *out_resid,
                 size_t ws_bytes);
sd_status allrows_launch(const void *target, const void *draft, sd_dtype dt,
                         long long d_seq_rows, const int32_t *tokens,
                         const float *uniforms, int B, int gamma, int V,
                         float T, int32_t *n_acc, int32_t *out_tokens,
                         float *out_prob, float *out_accept,
                         int32_t *dev_status, void *ws, size_t ws_bytes,
                         cudaStream_t stream);

// The fused fan-out's arguments (host F, device outputs).
struct FanArgs {
  const int32_t *F;  // [gamma + 1]
  int32_t *fan_tokens;
  float *fan_logit;
};

// The cluster size of the FAN kernels for these sizes (aligned rows: the
// rule of cluster_launch).
static int fan_cluster(int B, int V, sd_dtype dt) {
  const long long nvec = V / (dt == SD_F32 ? 4 : 8);
  int CL = choose_cluster(nvec);
  if (B >= 128 && CL > 8 && tune(SD_TUNE_CLUSTER) == 0) CL = 8;
  return CL;
}

// Workspace of the fused verify + fan-out: the work and row counters, the
// coverage marks, then the scans' records (24 bytes a thread a draft row;
// left out, and every row filtered whole, above 1 GB).
struct FanLayout {
  size_t fcov, cand_t, cand_i, cand_v, zero_end, total;
  bool records;
};
static FanLayout fan_layout(int B, int gamma, int V, sd_dtype dt) {
  auto r256 = [](size_t x) { return (x + 255) / 256 * 256; };
  FanLayout L;
  const size_t nb = B > 0 ? (size_t)B : 0;
  L.fcov = 256;
  L.zero_end = L.fcov + r256(nb * 4);
  const size_t nrec = nb * (size_t)(gamma > 0 ? gamma : 0) *
                      (size_t)fan_cluster(B, V, dt) * kThreads;
  L.cand_t = L.zero_end;
  L.cand_i = L.cand_t + r256(nrec * 4);
  L.cand_v = L.cand_i + r256(nrec * 4);
  L.total = L.cand_v + nrec * 16;
  L.records = nrec > 0 && L.total <= ((size_t)1 << 30);
  if (!L.records) L.total = L.zero_end;
  return L;
}
size_t fan_workspace(int B, int gamma, int V, sd_dtype dt) {
  return fan_layout(B, gamma, V, dt).total;
}

// Whether the fused kernel takes sd_verify_linear_fanout: 16-byte aligned
// rows through the ring.
bool fan_applicable(const void *target, const void *draft, sd_dtype dt,
                    int V) {
  const int eb = dt == SD_F32 ? 4 : 2;
  return aligned16(target) && aligned16(draft) && ((size_t)V * eb) % 16 == 0 &&
         tune(SD_TUNE_NO_TMA) == 0;
}

static sd_status cluster_launch(const void *target, const void *draft,
                                sd_dtype dt, long long d_seq_rows,
                                const int32_t *tokens, const float *uniforms,
                                int B, int gamma, int V, float T,
                                int32_t *n_acc, int32_t *out_tokens,
                                float *out_prob, float *out_accept,
                                float *out_resid, int32_t *dev_status,
                                void *ws, size_t ws_bytes,
                                cudaStream_t stream, const FanArgs *fan);

sd_status linear_launch(const void *target, const void *draft, sd_dtype dt,
                        long long d_seq_rows, const int32_t *tokens,
                        const float *uniforms, int B, int gamma, int V,
                        float T, int32_t *n_acc, int32_t *out_tokens,
                        float *out_prob, float *out_accept, float *out_resid,
                        int32_t *dev_status, void *ws, size_t ws_bytes,
                        cudaStream_t stream) {
  // small inputs: every row at once, then one decision per sequence
  // (sdv_allrows.cu), instead of a barrier and a decision per position
  if (use_allrows(B, gamma, V, dt, target, draft, T, out_resid, ws_bytes))
    return allrows_launch(target, draft, dt, d_seq_rows, tokens, uniforms, B,
                          gamma, V, T, n_acc, out_tokens, out_prob,
                          out_accept, dev_status, ws, ws_bytes, stream);
  return cluster_launch(target, draft, dt, d_seq_rows, tokens, uniforms, B,
                        gamma, V, T, n_acc, out_tokens, out_prob, out_accept,
                        out_resid, dev_status, ws, ws_bytes, stream, nullptr);
}

// The verify fused with the fan-out of the draft tensor [B, gamma + 1, V]
// (fan_applicable must hold; ws of fan_workspace(B) bytes at least).
sd_status linear_fan_launch(const void *target, const void *draft,
                            sd_dtype dt, const int32_t *tokens,
                            const float *uniforms, int B, int gamma, int V,
                            float T, const int32_t *F, int32_t *n_acc,
                            int32_t *out_tokens, float *out_prob,
                            int32_t *fan_tokens, float *fan_logit,
                            int32_t *dev_status, void *ws, size_t ws_bytes,
                            cudaStream_t stream) {
  const FanArgs fa{F, fan_tokens, fan_logit};
  return cluster_launch(target, draft, dt, gamma + 1, tokens, uniforms, B,
                        gamma, V, T, n_acc, out_tokens, out_prob, nullptr,
                        nullptr, dev_status, ws, ws_bytes, stream, &fa);
}

static sd_status cluster_launch(const void *target, const void *draft,
                                sd_dtype dt, long long d_seq_rows,
                                const int32_t *tokens, const float *uniforms,
                                int B, int gamma, int V, float T,
                                int32_t *n_acc, int32_t *out_tokens,
                                float *out_prob, float *out_accept,
                                float *out_resid, int32_t *dev_status,
                                void *ws, size_t ws_bytes,
                                cudaStream_t stream, const FanArgs *fan) {
  int sms = 0;
  sd_status st = check_device(&sms);
  if (st != SD_OK) return st;
  const bool greedy = (T == 0.f);
  const int eb = dt == SD_F32 ? 4 : 2, vw = dt == SD_F32 ? 4 : 8;
  const bool vec = aligned16(target) && (greedy || gamma == 0 ||
                                         aligned16(draft)) &&
                   ((size_t)V * eb) % 16 == 0;
  const int VW = vec ? vw : 1;
  const long long nvec = V / VW;
  // many sequences: smaller clusters keep more of them in flight (measured
  // on the 256 x 128256 fp32 workload: 8 beats 16)
  int CL = choose_cluster(nvec);
  if (B >= 128 && CL > 8 && tune(SD_TUNE_CLUSTER) == 0) CL = 8;
  const bool ring = vec && tune(SD_TUNE_NO_TMA) == 0;
  const long long per_cta = (nvec + CL - 1) / CL;
  const size_t seg_bytes = ((size_t)((per_cta + 31) / 32) * 4 + 127) / 128 * 128;
  const size_t smem = seg_bytes + (ring ? (size_t)kRingBytes : 0);
  if (smem > 96 * 1024)
    return fail(SD_ERR_UNSUPPORTED, "V=%d needs %zu B of shared memory", V,
                smem);
  if (fan && !ring)
    return fail(SD_ERR_UNSUPPORTED, "the fused fan-out needs aligned rows");
  LinearKernel kern = fan ? pick_linear_fan(dt, greedy)
                          : pick_linear(dt, vec, ring, greedy);
  int maxc = 0;
  st = max_active_clusters((const void *)kern, CL, smem, &maxc);
  if (st != SD_OK) return st;
  // fused fan-out: every resident cluster, those without a sequence take
  // fan-out rows from the start
  const int nclusters = (B < maxc && !fan) ? B : maxc;
  // helping, in the tail of the work counter only (measured at B = 8..64
  // sequences of 128256 fp32 columns: extra clusters helping from the start
  // slowed the owners down by 5-16 %; at B = 128 and 256 helping in the
  // tail took 2-6 % off)
  const size_t hws = help_workspace(B, gamma);
  const bool helpers = !fan && tune(SD_TUNE_HELPERS) != 0 && B > nclusters &&
                       hws != 0 && ws && ws_bytes >= hws &&
                       CL <= kHelpRanks && nclusters <= kHelpMaxClusters;
  LinearParams prm;
  prm.target = target;
  prm.draft = draft;
  prm.tokens = tokens;
  prm.uniforms = uniforms;
  prm.B = B;
  prm.gamma = gamma;
  prm.V = V;
  prm.d_seq_rows = d_seq_rows;
  prm.k2 = greedy ? 0.f : (float)(1.4426950408889634 / (double)T);
  prm.n_acc = n_acc;
  prm.out_tokens = out_tokens;
  prm.out_prob = out_prob;
  prm.out_accept = out_accept;
  prm.out_resid = out_resid;
  prm.dev_status = dev_status;
  prm.queue = nullptr;
  prm.nclusters = nclusters;
  prm.seg_bytes = (int)seg_bytes;
  prm.slice_vecs = (int)per_cta;
  prm.spec = tune(SD_TUNE_SPEC);
  prm.helping = prm.active = prm.opos = prm.hpos = prm.hflag = nullptr;
  prm.hpart = nullptr;
  prm.fan_tokens = nullptr;
  prm.fan_logit = nullptr;
  prm.ftotal = 0;
  prm.fq = nullptr;
  prm.fcov = nullptr;
  prm.cand_t = nullptr;
  prm.cand_i = nullptr;
  prm.cand_v = nullptr;
  if (fan) {
    const FanLayout L = fan_layout(B, gamma, V, dt);
    if (!ws || ws_bytes < L.zero_end)
      return fail(SD_ERR_INVALID_ARG, "workspace of >= %zu bytes required",
                  L.total);
    int o = 0;
    for (int k = 0; k <= gamma; ++k) {
      prm.fF[k] = fan->F[k];
      prm.foff[k] = o;
      o += fan->F[k];
    }
    prm.ftotal = o;
    prm.fan_tokens = fan->fan_tokens;
    prm.fan_logit = fan->fan_logit;
    char *w = static_cast<char *>(ws);
    prm.fq = reinterpret_cast<int *>(w + 4);
    // the records, when the workspace holds them for this cluster size
    if (!greedy && L.records && ws_bytes >= L.total &&
        fan_cluster(B, V, dt) == CL) {
      prm.fcov = reinterpret_cast<int *>(w + L.fcov);
      prm.cand_t = reinterpret_cast<float *>(w + L.cand_t);
      prm.cand_i = reinterpret_cast<int *>(w + L.cand_i);
      prm.cand_v = reinterpret_cast<uint4 *>(w + L.cand_v);
    }
  }
  if (B > nclusters) {
    if (!ws || ws_bytes < 256)
      return fail(SD_ERR_INVALID_ARG, "workspace of >= 256 bytes required");
    prm.queue = static_cast<int *>(ws);
  }
  if (helpers) {
    const HelpLayout L = help_layout(B, gamma);
    char *w = static_cast<char *>(ws);
    prm.helping = reinterpret_cast<int *>(w + 4);
    prm.active = reinterpret_cast<int *>(w + L.active);
    prm.opos = reinterpret_cast<int *>(w + L.opos);
    prm.hpos = reinterpret_cast<int *>(w + L.hpos);
    prm.hflag = reinterpret_cast<int *>(w + L.hflag);
    prm.hpart = reinterpret_cast<uint4 *>(w + L.hpart);
    SDV_CUDA(cudaMemsetAsync(ws, 0, L.zero_end, stream));
  } else if (fan) {
    SDV_CUDA(cudaMemsetAsync(ws, 0, fan_layout(B, gamma, V, dt).zero_end,
                             stream));
  } else if (prm.queue) {
    SDV_CUDA(cudaMemsetAsync(ws, 0, sizeof(int), stream));
  }
  void *args[] = {&prm};
  return launch_clusters((const void *)kern, nclusters, CL, smem, stream,
                         args);
}

}  // namespace sdv

extern "C" size_t sd_verify_linear_workspace(int B, int gamma, int V,
                                             sd_dtype dt) {
  // the work counter and, up to 768 KB, the helping records; wherever the
  // all-rows path could be taken (at any setting of SD_TUNE_ALLROWS), its
  // slice states (at most 512 KB)
  const size_t a = sdv::allrows_workspace(B, gamma, V, dt);
  const size_t h = sdv::help_workspace(B, gamma);
  const size_t w = a > h ? a : h;
  return w > 256 ? w : 256;
}

extern "C" sd_status sd_verify_linear(
    const void *target_logits, const void *draft_logits, sd_dtype dt,
    const int32_t *draft_tokens, const float *uniforms, int B, int gamma,
    int V, float T, int32_t *n_accepted, int32_t *out_tokens, float *out_prob,
    float *out_accept_prob, float *out_resid, int32_t *dev_status,
    void *workspace, size_t ws_bytes, void *stream) {
  SDV_REQUIRE(dt == SD_F32 || dt == SD_BF16, "bad dtype %d", (int)dt);
  SDV_REQUIRE(B >= 0, "B < 0");
  SDV_REQUIRE(gamma >= 0 && gamma <= SD_MAX_GAMMA, "gamma=%d outside [0, %d]",
              gamma, SD_MAX_GAMMA);
  SDV_REQUIRE(V >= 1 && V <= SD_MAX_V, "V=%d outside [1, %d]", V, SD_MAX_V);
  SDV_REQUIRE(T >= 0.f && std::isfinite(T), "T must be finite and >= 0");
  if (B == 0) return SD_OK;
  SDV_REQUIRE(target_logits && n_accepted && out_tokens, "null pointer");
  SDV_REQUIRE(gamma == 0 || draft_tokens, "draft_tokens is null");
  SDV_REQUIRE(T == 0.f || uniforms, "uniforms is null");
  SDV_REQUIRE(T == 0.f || gamma == 0 || draft_logits,
              "draft_logits is null with T > 0");
  return sdv::linear_launch(target_logits, draft_logits, dt, gamma,
                            draft_tokens, uniforms, B, gamma, V, T,
                            n_accepted, out_tokens, out_prob, out_accept_prob,
                            out_resid, dev_status, workspace, ws_bytes,
                            static_cast<cudaStream_t>(stream));
}
