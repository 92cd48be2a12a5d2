// sdv_kcand.cu -- K-candidate verify with verifier self-selection
// (SpecDiff-2, "core method": K joint drafts sampled from the drafter's
// position-wise marginals, all verified, the longest accepted streak kept).
// Rows that are 16-byte aligned go to the streaming kernel of
// sdv_kcand_ring.cu; this file's kernel (plain loads) takes the rest.
//
// One cluster verifies one sequence b at a time.  Position j is one step:
// the CTAs stream their slices of the shared draft marginal row (b, j) and
// of the target row (b, k, j) of every candidate still alive, exchange the
// per-row (max, sum) partials through distributed shared memory, and every
// CTA applies the accept test r <= p(x)/q(x) of each live candidate.  A
// candidate leaves at its first rejection; the scan stops when none is
// left, so rows past the last live candidate are never read.  The
// candidate with the most accepted tokens (lowest k on ties) gets the
// correction (its rejection pair, re-read from L2) or the bonus (its row
// gamma) by the cluster-wide inverse-CDF draw.
#include "sdv_device.cuh"
#include "sdv_host.cuh"

namespace sdv {

struct KcandParams {
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
};

constexpr int kMaxRows = SD_MAX_K + 1;  // draft row + one per candidate

struct KcandSmem {
  MS red[2][kWarps];
  AM ared[kWarps];
  MS part[2][kMaxRows];   // [parity][row] (peers read)
  AM apart[2][kMaxRows];
  MS mrg[kMaxRows];       // merged stats of this step's rows
  AM amrg[kMaxRows];
  int rowk[kMaxRows];     // candidate of row r (row 0: draft)
  int nrows;
  // per candidate
  int gx[SD_MAX_K];
  float gzt[SD_MAX_K], gzd[SD_MAX_K], gr[SD_MAX_K];
  int n_k[SD_MAX_K];
  MS rej_t[SD_MAX_K], rej_d[SD_MAX_K];  // stats at the rejection position
  int rej_am[SD_MAX_K];                 // greedy: argmax there
  unsigned alive, accept_mask;
  int invalid, bad_token;
  int next_seq[2];
  DrawSmem draw;
};

template <int DT, int VW, bool GREEDY>
__global__ void __launch_bounds__(kThreads, 2)
    kcand_verify_kernel(const KcandParams p) {
  extern __shared__ __align__(128) unsigned char dsm[];
  float *segmass = reinterpret_cast<float *>(dsm);
  __shared__ KcandSmem sh;
  using Row = GRow<DT, VW>;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank(), CL = (int)cluster.num_blocks();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = p.V, K = p.K, gamma = p.gamma, G1 = gamma + 1;
  const Slice sl = make_slice(V / VW, rank, CL);
  const size_t rowb = (size_t)V * elt_bytes<DT>();
  const char *tbase = static_cast<const char *>(p.target);
  const char *dbase = static_cast<const char *>(p.draft);
  const float k2 = p.k2;
  auto trow_of = [&](int b, int k, int j) {
    return tbase + (((size_t)b * K + k) * G1 + j) * rowb;
  };
  auto drow_of = [&](int b, int j) {
    return dbase + ((size_t)b * gamma + j) * rowb;
  };

  int par = 0, seqpar = 0;
  int b = (int)(blockIdx.x / CL);
  while (b < p.B) {
    if (tid == 0) {
      if (rank == 0)
        sh.next_seq[seqpar] =
            p.queue ? p.nclusters + atomicAdd(p.queue, 1) : p.B;
      sh.alive = K == 32 ? 0xffffffffu : ((1u << K) - 1u);
      sh.invalid = 0;
      sh.bad_token = 0;
    }
    if (tid < K) sh.n_k[tid] = gamma;
    __syncthreads();
    // ---------------- scan positions while a candidate is alive ----------
    for (int j = 0; j < gamma; ++j) {
      const unsigned alive = sh.alive;
      if (!alive) break;
      if (tid == 0) {
        int r = 0;
        if (!GREEDY) sh.rowk[r++] = -1;
        for (int k = 0; k < K; ++k)
          if (alive >> k & 1u) sh.rowk[r++] = k;
        sh.nrows = r;
      }
      if (tid < K && (alive >> tid & 1u)) {  // gathers for the accept tests
        const int k = tid;
        const int x = p.tokens[((size_t)b * K + k) * gamma + j];
        float zt = 0.f, zd = 0.f;
        if (!GREEDY && x >= 0 && x < V) {
          zt = load_logit<DT>(trow_of(b, k, j), x);
          zd = load_logit<DT>(drow_of(b, j), x);
        }
        sh.gx[k] = x;
        sh.gzt[k] = zt;
        sh.gzd[k] = zd;
        sh.gr[k] = GREEDY ? 0.f : p.uniforms[((size_t)b * K + k) * G1 + j];
      }
      __syncthreads();
      const int nrows = sh.nrows;
      auto row_ptr = [&](int r) {
        const int k = sh.rowk[r];
        return k < 0 ? drow_of(b, j) : trow_of(b, k, j);
      };
      // stream the rows two at a time
      for (int r0 = 0; r0 < nrows; r0 += 2) {
        const bool two = r0 + 1 < nrows;
        const Row ra{row_ptr(r0)};
        const Row rb{two ? row_ptr(r0 + 1) : row_ptr(r0)};
        if constexpr (GREEDY) {
          AM a = am_empty(), c = am_empty();
          argmax_pass<DT, VW>(ra, sl, a);
          a = block_reduce_am(a, sh.ared);
          if (tid == 0) sh.apart[par][r0] = a;
          if (two) {
            __syncthreads();  // the scratch of the first reduction is free
            argmax_pass<DT, VW>(rb, sl, c);
            c = block_reduce_am(c, sh.ared);
            if (tid == 0) sh.apart[par][r0 + 1] = c;
          }
        } else {
          MS st[2] = {ms_empty(), ms_empty()};
          stats_pass<DT, VW>(ra, rb, two, sl, k2, st[0], st[1]);
          block_reduce_ms<2>(st, k2, sh.red);
          if (tid == 0) {
            sh.part[par][r0] = st[0];
            if (two) sh.part[par][r0 + 1] = st[1];
          }
        }
        __syncthreads();
      }
      cluster.sync();
      // merge every row over the cluster (warp w: rows w, w+8, ...)
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
      par ^= 1;
      __syncthreads();
      // accept tests, one thread per live candidate
      if (warp == 0) {
        bool acc = false, bad = false, inv = false;
        const int k = lane;
        if (k < K && (alive >> k & 1u)) {
          int r = 0;  // row of candidate k
          for (int q = 0; q < nrows; ++q)
            if (sh.rowk[q] == k) r = q;
          const int x = sh.gx[k];
          bad = x < 0 || x >= V;
          if constexpr (GREEDY) {
            const AM a = sh.amrg[r];
            inv = a.bad || !(a.v > -kInf);
            acc = !inv && x == a.i;
            if (!acc) sh.rej_am[k] = a.i;
          } else {
            const MS mt = sh.mrg[r], md = sh.mrg[0];
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
        if (lane == 0) {
          sh.alive = am;  // candidates still alive after position j
          if (bm) sh.bad_token = 1;
          if (im) sh.invalid = 1;
        }
      }
      __syncthreads();
      if (sh.invalid) break;
    }
    // --------------------------- selection and final token ---------------
    const bool invalid = sh.invalid;
    int nsel = -1, ksel = -1;
    if (!invalid) {
      for (int k = 0; k < K; ++k)
        if (sh.n_k[k] > nsel) {
          nsel = sh.n_k[k];
          ksel = k;
        }
    }
    int t = -1;
    float prob = 0.f;
    bool inv_final = false;
    int zero_mass = 0;
    bool writer = (rank == 0 && warp == 0);
    if (!invalid) {
      const bool bonus = (nsel == gamma);
      const char *trow = trow_of(b, ksel, nsel);
      const char *drow = bonus ? nullptr : drow_of(b, nsel);
      MS mt = bonus ? ms_empty() : sh.rej_t[ksel];
      const MS md = bonus ? ms_empty() : sh.rej_d[ksel];
      int gt = GREEDY && !bonus ? sh.rej_am[ksel] : -1;
      if (bonus) {  // one more step: target row gamma of the selection
        const Row ra{trow};
        if constexpr (GREEDY) {
          AM a = am_empty();
          argmax_pass<DT, VW>(ra, sl, a);
          a = block_reduce_am(a, sh.ared);
          if (tid == 0) sh.apart[par][0] = a;
        } else {
          MS st[2] = {ms_empty(), ms_empty()};
          stats_pass<DT, VW>(ra, ra, false, sl, k2, st[0], st[1]);
          block_reduce_ms<2>(st, k2, sh.red);
          if (tid == 0) sh.part[par][0] = st[0];
        }
        cluster.sync();
        if (warp == 0) {
          if constexpr (GREEDY) {
            AM a = am_empty();
            if (lane < CL) a = cluster.map_shared_rank(&sh, lane)->apart[par][0];
            a = warp_down_am(a);
            if (lane == 0) sh.amrg[0] = a;
          } else {
            MS m = ms_empty();
            if (lane < CL) m = cluster.map_shared_rank(&sh, lane)->part[par][0];
            m = warp_down_ms(m, k2);
            if (lane == 0) sh.mrg[0] = m;
          }
        }
        par ^= 1;
        __syncthreads();
        if constexpr (GREEDY) {
          const AM a = sh.amrg[0];
          inv_final = a.bad || !(a.v > -kInf);
          gt = a.i;
        } else {
          mt = sh.mrg[0];
          inv_final = !ms_valid(mt);
        }
      }
      if (!inv_final) {
        if constexpr (GREEDY) {
          t = gt;
          prob = 1.f;
        } else {
          Weight W;
          W.k2 = k2;
          W.mtk = mt.m * k2;
          W.ist = 1.f / mt.s;
          W.mdk = md.m * k2;
          W.cq = 1.f / md.s;
          const float u = p.uniforms[((size_t)b * K + ksel) * G1 + gamma];
          const Row ra{trow}, rb{drow ? drow : trow};
          DrawOut o = cluster_draw<DT, VW>(cluster, sh.draw, segmass, ra, rb,
                                           !bonus, W, sl, u, par);
          if (o.owner < 0) {  // zero residual mass: draw from p instead
            zero_mass = 1;
            __syncthreads();
            o = cluster_draw<DT, VW>(cluster, sh.draw, segmass, ra, rb, false,
                                     W, sl, u, par);
          }
          writer = (o.owner == rank && warp == 0);
          t = o.t;
          prob = (float)((double)o.wt / o.N);
        }
      }
    }
    const bool bad_seq = invalid || inv_final;
    if (writer) {
      const int G = gamma;
      for (int i = lane; i <= G; i += 32) {
        int v = -1;
        if (!bad_seq) {
          if (i < nsel) v = p.tokens[((size_t)b * K + ksel) * G + i];
          else if (i == nsel) v = t;
        }
        p.out_tokens[(size_t)b * (G + 1) + i] = v;
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
    b = cluster.map_shared_rank(&sh, 0)->next_seq[seqpar];
    seqpar ^= 1;
    __syncthreads();
  }
  cluster.sync();
}

size_t kcand_help_workspace(int B, int K, int gamma);
sd_status kcand_ring_launch(const void *target, const void *draft,
                            sd_dtype dt, const int32_t *tokens,
                            const float *uniforms, int B, int K, int gamma,
                            int V, float T, int32_t *n_acc, int32_t *sel_k,
                            int32_t *out_tokens, int32_t *n_per_cand,
                            float *out_prob, int32_t *dev_status, void *ws,
                            size_t ws_bytes, cudaStream_t stream,
                            bool *launched);

using KcandKernel = void (*)(const KcandParams);

static KcandKernel pick_kcand(int dt, bool vec, bool greedy) {
  if (dt == SD_F32) {
    if (vec) return greedy ? kcand_verify_kernel<0, 4, true> : kcand_verify_kernel<0, 4, false>;
    return greedy ? kcand_verify_kernel<0, 1, true> : kcand_verify_kernel<0, 1, false>;
  }
  if (vec) return greedy ? kcand_verify_kernel<1, 8, true> : kcand_verify_kernel<1, 8, false>;
  return greedy ? kcand_verify_kernel<1, 1, true> : kcand_verify_kernel<1, 1, false>;
}

}  // namespace sdv

extern "C" size_t sd_verify_kcand_workspace(int B, int K, int gamma, int V,
                                            sd_dtype dt) {
  (void)V;
  (void)dt;
  // the work counter and, up to 64 MB, the helping records of the
  // streaming kernel (sdv_kcand_ring.cu)
  const size_t h = sdv::kcand_help_workspace(B, K, gamma);
  return h > 256 ? h : 256;
}

extern "C" sd_status sd_verify_kcand(
    const void *target_logits, const void *draft_logits, sd_dtype dt,
    const int32_t *draft_tokens, const float *uniforms, int B, int K,
    int gamma, int V, float T, int32_t *n_accepted, int32_t *selected_k,
    int32_t *out_tokens, int32_t *n_per_cand, float *out_prob,
    int32_t *dev_status, void *workspace, size_t ws_bytes, void *stream) {
  using namespace sdv;
  SDV_REQUIRE(dt == SD_F32 || dt == SD_BF16, "bad dtype %d", (int)dt);
  SDV_REQUIRE(B >= 0, "B < 0");
  SDV_REQUIRE(K >= 1 && K <= SD_MAX_K, "K=%d outside [1, %d]", K, SD_MAX_K);
  SDV_REQUIRE(gamma >= 0 && gamma <= SD_MAX_GAMMA, "gamma=%d outside [0, %d]",
              gamma, SD_MAX_GAMMA);
  SDV_REQUIRE(V >= 1 && V <= SD_MAX_V, "V=%d outside [1, %d]", V, SD_MAX_V);
  SDV_REQUIRE(T >= 0.f && std::isfinite(T), "T must be finite and >= 0");
  if (B == 0) return SD_OK;
  SDV_REQUIRE(target_logits && n_accepted && selected_k && out_tokens,
              "null pointer");
  SDV_REQUIRE(gamma == 0 || draft_tokens, "draft_tokens is null");
  SDV_REQUIRE(T == 0.f || uniforms, "uniforms is null");
  SDV_REQUIRE(T == 0.f || gamma == 0 || draft_logits,
              "draft_logits is null with T > 0");
  int sms = 0;
  sd_status st = check_device(&sms);
  if (st != SD_OK) return st;
  const bool greedy = (T == 0.f);
  const int eb = dt == SD_F32 ? 4 : 2, vw = dt == SD_F32 ? 4 : 8;
  const bool vec = aligned16(target_logits) &&
                   (greedy || gamma == 0 || aligned16(draft_logits)) &&
                   ((size_t)V * eb) % 16 == 0;
  if (vec) {  // 16-byte aligned rows: the streaming kernel
    bool launched = false;
    st = kcand_ring_launch(target_logits, draft_logits, dt, draft_tokens,
                           uniforms, B, K, gamma, V, T, n_accepted,
                           selected_k, out_tokens, n_per_cand, out_prob,
                           dev_status, workspace, ws_bytes,
                           static_cast<cudaStream_t>(stream), &launched);
    if (st != SD_OK || launched) return st;
  }
  const long long nvec = V / (vec ? vw : 1);
  const int CL = choose_cluster(nvec);
  const long long per_cta = (nvec + CL - 1) / CL;
  const size_t smem = ((size_t)((per_cta + 31) / 32) * 4 + 127) / 128 * 128;
  if (smem > 96 * 1024)
    return fail(SD_ERR_UNSUPPORTED, "V=%d needs %zu B of shared memory", V,
                smem);
  KcandKernel kern = pick_kcand(dt, vec, greedy);
  int maxc = 0;
  st = max_active_clusters((const void *)kern, CL, smem, &maxc);
  if (st != SD_OK) return st;
  const int nclusters = B < maxc ? B : maxc;
  KcandParams prm;
  prm.target = target_logits;
  prm.draft = draft_logits;
  prm.tokens = draft_tokens;
  prm.uniforms = uniforms;
  prm.B = B;
  prm.K = K;
  prm.gamma = gamma;
  prm.V = V;
  prm.k2 = greedy ? 0.f : (float)(1.4426950408889634 / (double)T);
  prm.n_acc = n_accepted;
  prm.sel_k = selected_k;
  prm.out_tokens = out_tokens;
  prm.n_per_cand = n_per_cand;
  prm.out_prob = out_prob;
  prm.dev_status = dev_status;
  prm.queue = nullptr;
  prm.nclusters = nclusters;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (B > nclusters) {
    if (!workspace || ws_bytes < 256)
      return fail(SD_ERR_INVALID_ARG, "workspace of >= 256 bytes required");
    prm.queue = static_cast<int *>(workspace);
    SDV_CUDA(cudaMemsetAsync(workspace, 0, sizeof(int), s));
  }
  void *args[] = {&prm};
  return launch_clusters((const void *)kern, nclusters, CL, smem, s, args);
}
