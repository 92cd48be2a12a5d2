// sdv_tree.cu -- token-tree verify (PRESTO, section 2.1: a token tree is
// verified prefix-wise from the root, the path's acceptance factorising
// along it; siblings are tried in turn with p <- norm(max(0, p - q)) after
// every rejection, the single-step residual of "01 · Draft-then-verify",
// section 2.1).
//
// One cluster walks one tree.  At the current node u the CTAs bring their
// slices of the target row p_u and the draft row q_u (which drafted u's
// children) into shared memory (TMA bulk copies when rows are 16-byte
// aligned), merge the (max, sum) partials, and try the children in
// increasing node index.  The repeated residual has a closed form: after k
// rejections the current distribution is max(0, p - c_k q) / N_k with
// c_0 = 0, N_0 = 1, c_{k+1} = c_k + N_k and N_{k+1} = sum max(0, p - c_{k+1} q)
// (max(0, max(0, p - c q)/N - q) = max(0, p - (c + N) q)/N because the left
// side vanishes wherever p <= c q).  So child v is accepted iff
//   U[v] <= max(0, p(t_v)/q(t_v) - c_k) / N_k,
// and each rejection costs one cluster-wide mass pass over the slices that
// are already in shared memory.  An accepted child becomes the current node;
// when every child is rejected, or at a leaf, the last token is drawn from
// the current distribution with uniform slot 0.  Only rows on the accepted
// path are read.
#include <type_traits>

#include "sdv_device.cuh"
#include "sdv_host.cuh"
#include "sdv_tma.cuh"

namespace sdv {

struct TreeParams {
  const void *target;  // [B, N, V]
  const void *draft;   // [B, N, V]
  const int32_t *parent;
  const int32_t *node_tokens;
  const float *uniforms;
  int B, N, V;
  float k2;
  int32_t *n_acc, *out_tokens, *out_nodes;
  // Optional row maps (null: node u reads row u of its sequence's N rows):
  // node u reads target row trow[b][u] of the sequence's trows rows and
  // draft row drow[b][u] of its drows rows.
  const int32_t *trow, *drow;
  int trows, drows;
  int out_cols;  // columns of out_tokens / out_nodes (<= N)
  const int32_t *node_cand;  // optional: out_cand[b] = node_cand of the
  int32_t *out_cand;         // last accepted node (0 when none)
  float *out_prob;
  int32_t *dev_status;
  int *queue;
  int nclusters;
  int seg_bytes, slice_vecs;
};

struct TreeSmem {
  MS red[2][kWarps];
  AM ared[kWarps];
  MS part[2][2];
  AM apart[2];
  MS mt, md;
  AM am;
  int invalid;
  int par_[SD_MAX_TREE_NODES];
  int tok[SD_MAX_TREE_NODES];
  float uni[SD_MAX_TREE_NODES];
  int kids[SD_MAX_TREE_NODES];
  float gzt[SD_MAX_TREE_NODES];
  union {
    float gzd[SD_MAX_TREE_NODES];  // draft logits of the children's tokens
    int ex[SD_MAX_TREE_NODES];     // deterministic drafts: removed tokens
  };
  int path[SD_MAX_TREE_NODES];
  int nkids;
  int next_seq[2];
  DrawSmem draw;
};

// Deterministic drafts.  The weights are p over the row without the
// removed tokens ex[0..ne).  mass_pass sums every token; the segments that
// hold a removed token are then summed again without them (one warp per
// segment), so every mass stays a sum of non-negative terms.
__device__ __forceinline__ bool is_removed(const int *ex, int ne, int j) {
  bool r = false;
  for (int i = 0; i < ne; ++i) r |= ex[i] == j;
  return r;
}

template <int DT, int VW, class Row>
__device__ __forceinline__ void det_weights(const Row &ra, const Weight &W,
                                            const int *ex, int ne, int v,
                                            float (&w)[VW]) {
  const Raw<DT, VW> a = ra.get(v);
  weights<DT, VW>(a, a, false, W, w);
#pragma unroll
  for (int e = 0; e < VW; ++e)
    if (is_removed(ex, ne, v * VW + e)) w[e] = 0.f;
}

template <int DT, int VW, class Row>
__device__ void det_fill(const Row &ra, const Weight &W, const Slice &sl,
                         float *segmass, const int *ex, int ne) {
  mass_pass<DT, VW>(ra, ra, false, W, sl, segmass);
  if (ne == 0) return;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  auto seg_of = [&](int j) {  // segment of token j in this slice, or -1
    const int v = j / VW;
    return (v >= sl.vbeg && v < sl.vend) ? (v - sl.vbeg) / 32 : -1;
  };
  for (int i = warp; i < ne; i += kWarps) {
    const int s = seg_of(ex[i]);
    bool first = s >= 0;  // the first removed token of its segment redoes it
    for (int r = 0; r < i && first; ++r) first = seg_of(ex[r]) != s;
    if (!first) continue;  // warp-uniform
    const int v = sl.vbeg + s * 32 + lane;
    float acc = 0.f;
    if (v < sl.vend) {
      float w[VW];
      det_weights<DT, VW>(ra, W, ex, ne, v, w);
#pragma unroll
      for (int e = 0; e < VW; ++e) acc += w[e];
    }
    acc = warp_down_sum(acc);
    if (lane == 0) segmass[s] = acc;
  }
}

template <int DT, int VW, class Row>
__device__ double det_mass(cg::cluster_group &cluster, DrawSmem &ds,
                           float *segmass, const Row &ra, const Weight &W,
                           const Slice &sl, const int *ex, int ne, float u,
                           int &par) {
  return cluster_total(cluster, ds, segmass, sl, u, par, [&] {
    det_fill<DT, VW>(ra, W, sl, segmass, ex, ne);
  });
}

// Inverse-CDF draw from p without the removed tokens (cluster-wide, every
// thread of every CTA calls it; see cluster_draw).
template <int DT, int VW, class Row>
__device__ DrawOut det_draw(cg::cluster_group &cluster, DrawSmem &ds,
                            float *segmass, const Row &ra, const Weight &W,
                            const Slice &sl, const int *ex, int ne, float u,
                            int &par) {
  det_mass<DT, VW>(cluster, ds, segmass, ra, W, sl, ex, ne, u, par);
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
        det_weights<DT, VW>(ra, W, ex, ne, v, w);
      } else {
#pragma unroll
        for (int e = 0; e < VW; ++e) w[e] = 0.f;
      }
      out.t = warp_pick<VW>(w, ds.tau_seg, (sl.vbeg + s * 32) * VW, &out.wt);
    }
  }
  return out;
}

template <int DT, int VW, bool GREEDY, bool TMA, bool DET>
__global__ void __launch_bounds__(kThreads, 2)
    tree_verify_kernel(const TreeParams p) {
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ TreeSmem sh;
  __shared__ uint64_t bar;
  using Row = std::conditional_t<TMA, SRow<DT, VW>, GRow<DT, VW>>;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank(), CL = (int)cluster.num_blocks();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = p.V, N = p.N;
  const Slice sl = make_slice(V / VW, rank, CL);
  const size_t rowb = (size_t)V * elt_bytes<DT>();
  const char *tbase = static_cast<const char *>(p.target);
  const char *dbase = static_cast<const char *>(p.draft);
  const float k2 = p.k2;
  float *segmass = reinterpret_cast<float *>(dsm);
  uint4 *tbuf = reinterpret_cast<uint4 *>(dsm + p.seg_bytes);
  uint4 *dbuf = tbuf + p.slice_vecs;
  const uint32_t slice_bytes = (uint32_t)(sl.vend - sl.vbeg) * 16u;
  uint32_t phase = 0;
  if (TMA) {
    if (tid == 0) {
      mbar_init(&bar, 1);
      fence_mbar_init();
    }
    __syncthreads();
  }
  auto row_of = [&](const char *g, uint4 *buf) {
    if constexpr (TMA) {
      (void)g;
      return Row{buf, sl.vbeg};
    } else {
      (void)buf;
      return Row{g};
    }
  };

  int par = 0, seqpar = 0;
  int b = (int)(blockIdx.x / CL);
  while (b < p.B) {
    if (rank == 0 && tid == 0)
      sh.next_seq[seqpar] =
          p.queue ? p.nclusters + atomicAdd(p.queue, 1) : p.B;
    // the tree's parent array, tokens and uniforms -> shared memory, and
    // the parent-array check (every CTA reads the same values)
    int bad = 0;
    for (int v = tid; v < N; v += kThreads) {
      const int pv = p.parent[(size_t)b * N + v];
      sh.par_[v] = pv;
      sh.tok[v] = p.node_tokens[(size_t)b * N + v];
      sh.uni[v] = GREEDY ? 0.f : p.uniforms[(size_t)b * N + v];
      bad |= (v == 0) ? (pv != -1) : (pv < 0 || pv >= v);
    }
    const bool bad_parent = __syncthreads_or(bad);
    int depth = 0, cur = 0, t = -1, kind = 0;  // kind 3: unusable row
    int bad_token = 0, zero_mass = 0;
    float prob = 0.f;
    bool writer = (rank == 0 && warp == 0);
    while (!bad_parent) {
      // children of cur in increasing node index (warp 0 compacts them)
      if (warp == 0) {
        int cnt = 0;
        for (int v0 = cur + 1; v0 < N; v0 += 32) {
          const int v = v0 + lane;
          const bool is = v < N && sh.par_[v] == cur;
          const unsigned m = __ballot_sync(0xffffffffu, is);
          if (is) sh.kids[cnt + __popc(m & ((1u << lane) - 1u))] = v;
          cnt += __popc(m);
        }
        if (lane == 0) sh.nkids = cnt;
      }
      __syncthreads();
      const int nk = sh.nkids;
      const bool has_q = (!GREEDY) && (!DET) && nk > 0;
      const size_t tr_i =
          p.trow ? (size_t)b * p.trows + p.trow[(size_t)b * N + cur]
                 : (size_t)b * N + cur;
      const size_t dr_i =
          p.drow ? (size_t)b * p.drows + max(p.drow[(size_t)b * N + cur], 0)
                 : (size_t)b * N + cur;
      const char *trow = tbase + tr_i * rowb;
      const char *drow = dbase + dr_i * rowb;
      if (TMA && tid == 0) {
        fence_proxy_async();
        mbar_expect_tx(&bar, slice_bytes * (has_q ? 2u : 1u));
        if (slice_bytes) {
          bulk_g2s(tbuf, trow + (size_t)sl.vbeg * 16, slice_bytes, &bar);
          if (has_q) bulk_g2s(dbuf, drow + (size_t)sl.vbeg * 16, slice_bytes, &bar);
        }
      }
      // gathers of the children's logits (used after the merge)
      for (int i = tid; i < nk; i += kThreads) {
        const int x = sh.tok[sh.kids[i]];
        float zt = 0.f, zd = 0.f;
        if (!GREEDY && x >= 0 && x < V) {
          zt = load_logit<DT>(trow, x);
          if (!DET) zd = load_logit<DT>(drow, x);
        }
        sh.gzt[i] = zt;
        if (!DET) sh.gzd[i] = zd;
      }
      if (TMA) {
        mbar_wait(&bar, phase, p.dev_status);
        phase ^= 1;
      }
      const Row ra = row_of(trow, tbuf), rb = row_of(drow, dbuf);
      if constexpr (GREEDY) {
        AM a = am_empty();
        argmax_pass<DT, VW>(ra, sl, a);
        a = block_reduce_am(a, sh.ared);
        if (tid == 0) sh.apart[par] = a;
      } else {
        MS st[2] = {ms_empty(), ms_empty()};
        stats_pass<DT, VW>(ra, rb, has_q, sl, k2, st[0], st[1]);
        block_reduce_ms<2>(st, k2, sh.red);
        if (tid == 0) {
          sh.part[par][0] = st[0];
          sh.part[par][1] = st[1];
        }
      }
      cluster.sync();
      if (warp == 0) {
        if constexpr (GREEDY) {
          AM a = am_empty();
          if (lane < CL) a = cluster.map_shared_rank(&sh, lane)->apart[par];
          a = warp_down_am(a);
          if (lane == 0) {
            sh.am = a;
            sh.invalid = a.bad || !(a.v > -kInf);
          }
        } else {
          MS mt = ms_empty(), md = ms_empty();
          if (lane < CL) {
            const TreeSmem *rs = cluster.map_shared_rank(&sh, lane);
            mt = rs->part[par][0];
            md = rs->part[par][1];
          }
          mt = warp_down_ms(mt, k2);
          md = warp_down_ms(md, k2);
          if (lane == 0) {
            sh.mt = mt;
            sh.md = md;
            sh.invalid = !ms_valid(mt) || (has_q && !ms_valid(md));
          }
        }
      }
      par ^= 1;
      __syncthreads();
      if (sh.invalid) {
        kind = 3;
        break;
      }
      for (int i = 0; i < nk; ++i) {
        const int x = sh.tok[sh.kids[i]];
        if (x < 0 || x >= V) bad_token = 1;
      }
      int next = -1;
      if constexpr (GREEDY) {
        const int a = sh.am.i;
        for (int i = 0; i < nk && next < 0; ++i)
          if (sh.tok[sh.kids[i]] == a) next = sh.kids[i];
        if (next < 0) {
          t = a;
          prob = 1.f;
          break;
        }
      } else if constexpr (DET) {
        // deterministic drafts: child v is accepted iff U[v] <= p'(t_v),
        // p' = p outside the tokens removed so far (sh.ex), renormalised
        Weight W;
        W.k2 = k2;
        W.mtk = sh.mt.m * k2;
        W.ist = 1.f / sh.mt.s;
        W.mdk = 0.f;
        W.cq = 0.f;
        int ne = 0;
        double Nr = 1.0;  // mass of p outside the removed tokens
        bool zm = false;
        for (int i = 0; i < nk; ++i) {
          const int v = sh.kids[i];
          const int x = sh.tok[v];
          if (x < 0 || x >= V) continue;  // rejected, removes nothing
          bool removed = false;
          for (int r = 0; r < ne; ++r) removed |= sh.ex[r] == x;
          const float wx =
              removed ? 0.f
                      : __fmul_rn(ex2(fmaf(sh.gzt[i], k2, -W.mtk)), W.ist);
          const float rho = (float)((double)wx / Nr);
          if (sh.uni[v] <= rho) {
            next = v;
            break;
          }
          if (removed) continue;
          if (tid == 0) sh.ex[ne] = x;
          ++ne;
          if (i + 1 < nk) {  // (the final draw forms its own mass)
            if ((double)wx <= 0.5 * Nr) {
              // a minor token: N - w(x) loses at most a factor 2 of
              // relative precision, and no pass or cluster barrier is
              // needed (every CTA subtracts the same w(x))
              Nr -= (double)wx;
              __syncthreads();  // sh.ex[ne - 1] is seen by every thread
            } else {  // a dominant one: sum the rest again
              __syncthreads();
              Nr = det_mass<DT, VW>(cluster, sh.draw, segmass, ra, W, sl,
                                    sh.ex, ne, -1.f, par);
              __syncthreads();
              if (!(Nr > 0.0)) {
                zm = true;
                break;
              }
            }
          }
        }
        if (next < 0) {
          __syncthreads();
          const float u = sh.uni[0];
          DrawOut o = det_draw<DT, VW>(cluster, sh.draw, segmass, ra, W, sl,
                                       sh.ex, zm ? 0 : ne, u, par);
          if (o.owner < 0) {
            zm = true;
            __syncthreads();
            o = det_draw<DT, VW>(cluster, sh.draw, segmass, ra, W, sl, sh.ex,
                                 0, u, par);
          }
          zero_mass = zm;
          writer = (o.owner == rank && warp == 0);
          t = o.t;
          prob = (float)((double)o.wt / o.N);
          break;
        }
      } else {
        const MS mt = sh.mt, md = sh.md;
        Weight W;
        W.k2 = k2;
        W.mtk = mt.m * k2;
        W.ist = 1.f / mt.s;
        W.mdk = md.m * k2;
        double c = 0.0, Nc = 1.0;  // p^(k) = max(0, p - c q) / Nc
        bool zm = false;
        for (int i = 0; i < nk; ++i) {
          const int v = sh.kids[i];
          const int x = sh.tok[v];
          float rho = 0.f;
          if (x >= 0 && x < V) {
            const double ratio =
                (double)accept_ratio(sh.gzt[i], sh.gzd[i], mt, md, k2);
            rho = (float)(fmax(0.0, ratio - c) / Nc);
          }
          if (sh.uni[v] <= rho) {
            next = v;
            break;
          }
          // rejected: c <- c + N; N <- sum max(0, p - c q)
          c += Nc;
          if (i + 1 < nk) {
            W.cq = (float)(c / (double)md.s);
            Nc = cluster_mass<DT, VW>(cluster, sh.draw, segmass, ra, rb, true,
                                      W, sl, -1.f, par);
            __syncthreads();
            if (!(Nc > 0.0)) {
              zm = true;
              break;
            }
          }
        }
        if (next < 0) {
          // the last token: from max(0, p - c q) (or p at a leaf / after a
          // zero-mass residual)
          const bool use_q = has_q && !zm;
          W.cq = use_q ? (float)(c / (double)md.s) : 0.f;
          const float u = sh.uni[0];
          DrawOut o = cluster_draw<DT, VW>(cluster, sh.draw, segmass, ra, rb,
                                           use_q, W, sl, u, par);
          if (o.owner < 0) {
            zm = true;
            __syncthreads();
            o = cluster_draw<DT, VW>(cluster, sh.draw, segmass, ra, rb, false,
                                     W, sl, u, par);
          }
          zero_mass = zm;
          writer = (o.owner == rank && warp == 0);
          t = o.t;
          prob = (float)((double)o.wt / o.N);
          break;
        }
      }
      if (tid == 0) sh.path[depth] = next;
      ++depth;
      cur = next;
      __syncthreads();
    }
    const bool bad_seq = bad_parent || kind == 3;
    if (writer) {
      for (int i = lane; i < p.out_cols; i += 32) {
        int nd = -1, tk = -1;
        if (!bad_seq) {
          if (i < depth) {
            nd = sh.path[i];
            tk = sh.tok[nd];
          } else if (i == depth) {
            tk = t;
          }
        }
        if (p.out_nodes) p.out_nodes[(size_t)b * p.out_cols + i] = nd;
        p.out_tokens[(size_t)b * p.out_cols + i] = tk;
      }
      if (lane == 0) {
        p.n_acc[b] = bad_seq ? -1 : depth;
        if (p.out_cand)
          p.out_cand[b] =
              bad_seq ? -1
                      : (depth ? p.node_cand[(size_t)b * N +
                                             sh.path[depth - 1]]
                               : 0);
        if (p.out_prob) p.out_prob[b] = bad_seq ? 0.f : prob;
        status_or(p.dev_status,
                  (bad_token ? SD_DEV_BAD_TOKEN : 0) |
                      (bad_parent ? SD_DEV_BAD_PARENT : 0) |
                      (kind == 3 ? SD_DEV_NONFINITE : 0) |
                      (zero_mass ? SD_DEV_ZERO_MASS : 0));
      }
    }
    if (bad_parent) cluster.sync();  // keep next_seq visible to all CTAs
    b = cluster.map_shared_rank(&sh, 0)->next_seq[seqpar];
    seqpar ^= 1;
    __syncthreads();
  }
  cluster.sync();
}

using TreeKernel = void (*)(const TreeParams);

template <int DT, int VW, bool TMA>
static TreeKernel pick_tree_t(bool greedy, bool det) {
  if (greedy) return tree_verify_kernel<DT, VW, true, TMA, false>;
  return det ? tree_verify_kernel<DT, VW, false, TMA, true>
             : tree_verify_kernel<DT, VW, false, TMA, false>;
}

static TreeKernel pick_tree(int dt, bool vec, bool tma, bool greedy,
                            bool det) {
  if (dt == SD_F32) {
    if (!vec) return pick_tree_t<0, 1, false>(greedy, det);
    return tma ? pick_tree_t<0, 4, true>(greedy, det)
               : pick_tree_t<0, 4, false>(greedy, det);
  }
  if (!vec) return pick_tree_t<1, 1, false>(greedy, det);
  return tma ? pick_tree_t<1, 8, true>(greedy, det)
             : pick_tree_t<1, 8, false>(greedy, det);
}

constexpr size_t kTreeTmaSmemMax = 96 * 1024;


}  // namespace sdv

extern "C" size_t sd_verify_tree_workspace(int B, int N, int V, sd_dtype dt) {
  (void)B;
  (void)N;
  (void)V;
  (void)dt;
  return 256;
}

sd_status sdv::tree_launch(
    const void *target_logits, const void *draft_logits, sd_dtype dt,
    const int32_t *parent, const int32_t *node_tokens, const float *uniforms,
    int B, int N, int V, float T, bool det, int32_t *n_accepted,
    int32_t *out_tokens, int32_t *out_nodes, float *out_prob,
    int32_t *dev_status, void *workspace, size_t ws_bytes, void *stream,
    const sdv::TreeMaps *maps) {
  using namespace sdv;
  SDV_REQUIRE(dt == SD_F32 || dt == SD_BF16, "bad dtype %d", (int)dt);
  SDV_REQUIRE(B >= 0, "B < 0");
  SDV_REQUIRE(N >= 1, "N < 1");
  if (N > SD_MAX_TREE_NODES)
    return fail(SD_ERR_UNSUPPORTED, "N=%d above %d", N, SD_MAX_TREE_NODES);
  SDV_REQUIRE(V >= 1 && V <= SD_MAX_V, "V=%d outside [1, %d]", V, SD_MAX_V);
  SDV_REQUIRE(T >= 0.f && std::isfinite(T), "T must be finite and >= 0");
  if (B == 0) return SD_OK;
  SDV_REQUIRE(target_logits && parent && node_tokens && n_accepted &&
                  out_tokens && (out_nodes || maps),
              "null pointer");
  SDV_REQUIRE(T == 0.f || (uniforms && (det || draft_logits)),
              "uniforms and draft_logits are required when T > 0");
  int sms = 0;
  sd_status st = check_device(&sms);
  if (st != SD_OK) return st;
  const bool greedy = (T == 0.f);
  const int eb = dt == SD_F32 ? 4 : 2, vw = dt == SD_F32 ? 4 : 8;
  const bool one_row = greedy || det;  // no draft rows are read
  const bool vec = aligned16(target_logits) &&
                   (one_row || aligned16(draft_logits)) &&
                   ((size_t)V * eb) % 16 == 0;
  const long long nvec = V / (vec ? vw : 1);
  // Cluster size: the row-length rule, but a tree waiting for a free
  // cluster costs more than smaller slices do: when clusters of 16 cannot
  // all be resident for the B trees, clusters of 8 are used (measured on
  // 16 and 64 trees of 151936 bf16 columns: 24-36 % faster).
  int CL = choose_cluster(nvec);
  long long per_cta = 0;
  size_t seg_bytes = 0, smem = 0;
  bool tma = false;
  TreeKernel kern = nullptr;
  int maxc = 0;
  for (;;) {
    per_cta = (nvec + CL - 1) / CL;
    seg_bytes = ((size_t)((per_cta + 31) / 32) * 4 + 127) / 128 * 128;
    const size_t tma_smem =
        seg_bytes + (one_row ? 1 : 2) * (size_t)per_cta * 16;
    tma = vec && tma_smem <= kTreeTmaSmemMax && tune(SD_TUNE_NO_TMA) == 0;
    smem = tma ? tma_smem : seg_bytes;
    if (smem > 96 * 1024)
      return fail(SD_ERR_UNSUPPORTED, "V=%d needs %zu B of shared memory", V,
                  smem);
    kern = pick_tree(dt, vec, tma, greedy, det);
    st = max_active_clusters((const void *)kern, CL, smem, &maxc);
    if (st != SD_OK) return st;
    if (CL > 8 && maxc < B && tune(SD_TUNE_CLUSTER) == 0) {
      CL = 8;
      continue;
    }
    break;
  }
  const int nclusters = B < maxc ? B : maxc;
  TreeParams prm;
  prm.target = target_logits;
  prm.draft = draft_logits;
  prm.parent = parent;
  prm.node_tokens = node_tokens;
  prm.uniforms = uniforms;
  prm.B = B;
  prm.N = N;
  prm.V = V;
  prm.k2 = greedy ? 0.f : (float)(1.4426950408889634 / (double)T);
  prm.n_acc = n_accepted;
  prm.out_tokens = out_tokens;
  prm.out_nodes = out_nodes;
  prm.trow = maps ? maps->trow : nullptr;
  prm.drow = maps ? maps->drow : nullptr;
  prm.trows = maps ? maps->trows : N;
  prm.drows = maps ? maps->drows : N;
  prm.out_cols = maps ? maps->out_cols : N;
  prm.node_cand = maps ? maps->node_cand : nullptr;
  prm.out_cand = maps ? maps->out_cand : nullptr;
  prm.out_prob = out_prob;
  prm.dev_status = dev_status;
  prm.queue = nullptr;
  prm.nclusters = nclusters;
  prm.seg_bytes = (int)seg_bytes;
  prm.slice_vecs = (int)per_cta;
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

extern "C" sd_status sd_verify_tree(
    const void *target_logits, const void *draft_logits, sd_dtype dt,
    const int32_t *parent, const int32_t *node_tokens, const float *uniforms,
    int B, int N, int V, float T, int32_t *n_accepted, int32_t *out_tokens,
    int32_t *out_nodes, float *out_prob, int32_t *dev_status,
    void *workspace, size_t ws_bytes, void *stream) {
  return sdv::tree_launch(target_logits, draft_logits, dt, parent, node_tokens,
                          uniforms, B, N, V, T, false, n_accepted,
                          out_tokens, out_nodes, out_prob, dev_status,
                          workspace, ws_bytes, stream);
}

extern "C" size_t sd_verify_tree_det_workspace(int B, int N, int V,
                                               sd_dtype dt) {
  return sd_verify_tree_workspace(B, N, V, dt);
}

extern "C" sd_status sd_verify_tree_det(
    const void *target_logits, sd_dtype dt, const int32_t *parent,
    const int32_t *node_tokens, const float *uniforms, int B, int N, int V,
    float T, int32_t *n_accepted, int32_t *out_tokens, int32_t *out_nodes,
    float *out_prob, int32_t *dev_status, void *workspace, size_t ws_bytes,
    void *stream) {
  return sdv::tree_launch(target_logits, nullptr, dt, parent, node_tokens,
                          uniforms, B, N, V, T, true, n_accepted,
                          out_tokens, out_nodes, out_prob, dev_status,
                          workspace, ws_bytes, stream);
}
