// sdv_presto.cu -- device tree construction: one depth of PRESTO's beam
// search ("PRESTO", section 4.1: prefix-aligned score s_{d,t}(c_d) =
// log q_d(t) + lambda log rho_d(t | c_d), path score S(P) of Eq. 10;
// section 4.2 and Algorithm 1: beam search with global retention under a
// node budget; section 4.4: s is the log of the product of experts
// q rho^lambda up to a constant), and SpecBranch's branch resampling
// ("SpecBranch", branch resampling: k = max(1, floor(k_max (1 - q(x_b))))
// branches, the Top-k of the draft distribution at the branch point).
//
// Both are a top-b selection over a score row, then a small merge:
//  1. select: grid (sequence, path, slice).  Each CTA streams its slice of
//     the drafter's marginal row q_d (and of the path's log rho row) once
//     with 16-byte loads, forms v = z / T + lambda log rho per element, and
//     keeps the slice's b best (v, token) keys with the per-warp filters of
//     sdv_topf.cuh; it also keeps the online (max, sum) of q_d.
//  2. merge: one CTA per sequence ranks each path's slice lists into its
//     top-b, forms the candidates' path scores S + v - log sum exp(z / T),
//     orders them by (score desc, path asc, token asc) and appends them to
//     the tree while the node budget lasts; the first W become the next
//     frontier.  The fork's merge ranks the single row's lists into its
//     top-k_max and sizes k from q(x_b).
#include "sdv_device.cuh"
#include "sdv_host.cuh"
#include "sdv_topf.cuh"

namespace sdv {

constexpr int kPrestoMaxCand = 1024;  // W b per sequence (merge in smem)
constexpr int kPrestoMaxKeys = 1024;  // slices x b per path

struct SelParams {
  const void *q;        // row b at q + b * q_stride elements
  long long q_stride;
  const void *rho;      // [B, W, V] log rho (null: lambda == 0)
  int B, W, V, S;       // S slices per row
  float scale;          // v = z * scale + lambda * log rho
  float lambda;
  float k2;             // log2(e) / T for the (max, sum) of q
  int F;                // keys kept per slice
  const int32_t *frontier_node;  // [B, W] (null: every path active)
  const int32_t *n_nodes;        // [B] (null: every sequence active)
  int budget;
  uint64_t *keys;  // [B, W, S, F]
  MS *stats;       // [B, W, S]
  int *bad;        // [B, W, S]: a NaN or +inf was read
};

constexpr int kSelUF = 4;  // vectors of each row in flight per thread

template <int DT, int VW, bool RHO>
__global__ void __launch_bounds__(kThreads)
    presto_select_kernel(const SelParams p) {
  __shared__ TopSmem top;
  __shared__ MS red[1][kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int item = blockIdx.x / p.S, s = blockIdx.x % p.S;
  const int b = item / p.W, w = item % p.W;
  const size_t slot = (size_t)item * p.S + s;
  griddep_wait();  // the previous merge's tree state and keys are final
  const bool active =
      (!p.frontier_node || p.frontier_node[(size_t)b * p.W + w] >= 0) &&
      (!p.n_nodes || (p.n_nodes[b] >= 0 && p.n_nodes[b] < p.budget));
  if (!active) {  // block-uniform
    for (int i = tid; i < p.F; i += kThreads) p.keys[slot * p.F + i] = 0;
    if (tid == 0) {
      p.stats[slot] = ms_empty();
      p.bad[slot] = 0;
    }
    return;
  }
  const int nvec = p.V / VW;
  const Slice sl = make_slice(nvec, s, p.S);
  const char *qrow = static_cast<const char *>(p.q) +
                     (size_t)b * (size_t)p.q_stride * elt_bytes<DT>();
  const char *rrow =
      RHO ? static_cast<const char *>(p.rho) +
                ((size_t)b * p.W + w) * (size_t)p.V * elt_bytes<DT>()
          : nullptr;
  if (tid == 0) top.th = 0;
  __syncthreads();
  WarpFilter wf;
  wf_init(wf, p.F);
  MS st = ms_empty();
  float worst = -__builtin_huge_valf();  // NaN-propagating max of v
  for (int vb = sl.vbeg + warp * 32 * kSelUF; vb < sl.vend;
       vb += kWarps * 32 * kSelUF) {  // warp-uniform
    Raw<DT, VW> xq[kSelUF], xr[kSelUF];
#pragma unroll
    for (int u = 0; u < kSelUF; ++u) {
      const int v = vb + u * 32 + lane;
      if (v < sl.vend) {
        xq[u] = load_vec<DT, VW>(qrow, v);
        if (RHO) xr[u] = load_vec<DT, VW>(rrow, v);
      }
    }
    float z[kSelUF][VW];
#pragma unroll
    for (int u = 0; u < kSelUF; ++u) {
      const bool ok = vb + u * 32 + lane < sl.vend;
#pragma unroll
      for (int e = 0; e < VW; ++e) {
        float x = -__builtin_huge_valf();
        if (ok) {
          x = elt<DT, VW>(xq[u], e) * p.scale;
          if (RHO) x = fmaf(p.lambda, elt<DT, VW>(xr[u], e), x);
        }
        z[u][e] = x;
      }
      if (ok) {
        ms_add<DT, VW>(st, xq[u], p.k2);
        worst = max_nan(worst, vmax_nan_of<VW>(z[u]));
      }
    }
    if (!wf.seeded) {  // seed from the whole first batch (kSelUF VW values)
      float m1 = -__builtin_huge_valf(), m2 = -__builtin_huge_valf();
#pragma unroll
      for (int u = 0; u < kSelUF; ++u)
#pragma unroll
        for (int e = 0; e < VW; ++e) top2_add(m1, m2, z[u][e]);
      wf_seed2(wf, m1, m2);
    }
    wf_sync(wf, &top.th);
#pragma unroll
    for (int u = 0; u < kSelUF; ++u) {
      const int v = vb + u * 32 + lane;
      wf_offer_vals<VW>(wf, &top.th, z[u], v < sl.vend, v * VW);
    }
  }
  griddep_launch_dependents();  // the merge may start launching
  // a NaN anywhere, or +inf (in q, or in log rho), makes the row unusable
  const int anybad =
      __syncthreads_or(!(worst < __builtin_huge_valf()) &&
                       !(worst == -__builtin_huge_valf()));
  MS sts[1] = {st};
  block_reduce_ms<1>(sts, p.k2, red);
  wf_export(wf, top);
  __syncthreads();
  const int nout = rank_select(top, kWarps * p.F, p.F);
  for (int i = tid; i < p.F; i += kThreads)
    p.keys[slot * p.F + i] = i < nout ? top.out[i] : 0;
  if (tid == 0) {
    p.stats[slot] = sts[0];
    p.bad[slot] = anybad;
  }
}


// Rank the n keys of buf (0 = empty) and place the best F non-empty ones
// whose value is above -inf in out (descending); returns how many.
// Block-wide.
__device__ int rank_keys(const uint64_t *buf, int n, int F, uint64_t *out) {
  int cnt = 0;
  for (int i0 = 0; i0 < n; i0 += kThreads) {
    const int i = i0 + (int)threadIdx.x;
    const uint64_t me = i < n ? buf[i] : 0;
    const bool use = me != 0 && key_val(me) > -__builtin_huge_valf();
    if (use) {
      int r = 0;
      for (int j = 0; j < n; ++j) r += buf[j] > me;
      if (r < F) out[r] = me;
    }
    cnt += __syncthreads_count(use);
  }
  __syncthreads();
  return cnt < F ? cnt : F;
}

struct MergeParams {
  const uint64_t *keys;
  const MS *stats;
  const int *bad;
  int B, W, S, F;
  float k2, scale;
  int budget;
  int32_t *n_nodes, *parent, *node_tokens;
  float *node_score;
  int32_t *frontier_node;
  float *frontier_score;
  int32_t *dev_status;
};

struct Cand {
  float score;
  int w, tok;
};

__device__ __forceinline__ bool cand_better(const Cand &a, const Cand &b) {
  if (a.score != b.score) return a.score > b.score;
  if (a.w != b.w) return a.w < b.w;
  return a.tok < b.tok;
}

__global__ void __launch_bounds__(kThreads)
    presto_merge_kernel(const MergeParams p) {
  __shared__ uint64_t kbuf[kPrestoMaxKeys];
  __shared__ uint64_t best[SD_MAX_FANOUT];
  __shared__ Cand cand[kPrestoMaxCand];
  __shared__ int ofn[SD_MAX_FANOUT];
  __shared__ float ofs[SD_MAX_FANOUT];
  __shared__ float lse_s;
  __shared__ int invalid_s;
  const int tid = threadIdx.x;
  const int b = blockIdx.x;
  griddep_wait();  // every slice list of this depth is written
  griddep_launch_dependents();
  const int n0 = p.n_nodes[b];
  if (n0 < 0 || n0 >= p.budget) return;  // block-uniform
  const int W = p.W, S = p.S, F = p.F;
  for (int w = tid; w < W; w += kThreads) {
    ofn[w] = p.frontier_node[(size_t)b * W + w];
    ofs[w] = p.frontier_score[(size_t)b * W + w];
  }
  __syncthreads();
  if (tid == 0) {
    int bad = 0, w0 = -1;
    for (int w = 0; w < W; ++w) {
      if (ofn[w] < 0) continue;
      if (w0 < 0) w0 = w;
      for (int s = 0; s < S; ++s) bad |= p.bad[((size_t)b * W + w) * S + s];
    }
    float lse = 0.f;
    if (w0 >= 0) {
      MS a = ms_empty();
      for (int s = 0; s < S; ++s)
        a = ms_merge(a, p.stats[((size_t)b * W + w0) * S + s], p.k2);
      if (!ms_valid(a)) bad = 1;
      // log sum_j exp(z_j / T) = m / T + ln s
      lse = fmaf(a.m, p.scale, logf(a.s));
    }
    lse_s = lse;
    invalid_s = bad;
  }
  __syncthreads();
  if (invalid_s) {
    for (int w = tid; w < W; w += kThreads) {
      p.frontier_node[(size_t)b * W + w] = -1;
      p.frontier_score[(size_t)b * W + w] = 0.f;
    }
    if (tid == 0) {
      p.n_nodes[b] = -1;
      status_or(p.dev_status, SD_DEV_NONFINITE);
    }
    return;
  }
  const float lse = lse_s;
  // each path's top-F over its slices, as candidates in rank order
  int nc = 0;
  for (int w = 0; w < W; ++w) {  // block-uniform
    if (ofn[w] < 0) continue;
    const uint64_t *src = p.keys + ((size_t)b * W + w) * S * F;
    for (int i = tid; i < S * F; i += kThreads) kbuf[i] = src[i];
    __syncthreads();
    const int nb = rank_keys(kbuf, S * F, F, best);
    for (int i = tid; i < nb; i += kThreads) {
      Cand c;
      c.score = ofs[w] + (key_val(best[i]) - lse);
      c.w = w;
      c.tok = key_idx(best[i]);
      cand[nc + i] = c;
    }
    nc += nb;
    __syncthreads();
  }
  // order every candidate; the first min(nc, budget - n0) become nodes
  const int add = min(nc, p.budget - n0);
  for (int i = tid; i < nc; i += kThreads) {
    const Cand me = cand[i];
    int r = 0;
    for (int j = 0; j < nc; ++j) r += cand_better(cand[j], me);
    if (r < add) {
      const size_t v = (size_t)b * p.budget + n0 + r;
      p.parent[v] = ofn[me.w];
      p.node_tokens[v] = me.tok;
      p.node_score[v] = me.score;
    }
    if (r < W && r < add) {
      p.frontier_node[(size_t)b * W + r] = n0 + r;
      p.frontier_score[(size_t)b * W + r] = me.score;
    }
  }
  for (int w = add + tid; w < W; w += kThreads) {
    p.frontier_node[(size_t)b * W + w] = -1;
    p.frontier_score[(size_t)b * W + w] = 0.f;
  }
  if (tid == 0) p.n_nodes[b] = n0 + add;
}

struct ForkParams {
  const uint64_t *keys;
  const MS *stats;
  const int *bad;
  const void *draft;
  int dt;
  int B, V, S, F;
  float k2;
  int greedy;
  const int32_t *x_b;
  int32_t *out_k, *out_tokens;
  int32_t *dev_status;
};

__global__ void __launch_bounds__(kThreads)
    fork_merge_kernel(const ForkParams p) {
  __shared__ uint64_t kbuf[kPrestoMaxKeys];
  __shared__ uint64_t best[SD_MAX_FANOUT];
  __shared__ int k_s;
  const int tid = threadIdx.x;
  const int b = blockIdx.x;
  const int S = p.S, F = p.F;
  griddep_wait();  // every slice list is written
  for (int i = tid; i < S * F; i += kThreads)
    kbuf[i] = p.keys[(size_t)b * S * F + i];
  __syncthreads();
  const int nb = rank_keys(kbuf, S * F, F, best);
  if (tid == 0) {
    int bad = 0;
    MS a = ms_empty();
    for (int s = 0; s < S; ++s) {
      bad |= p.bad[(size_t)b * S + s];
      a = ms_merge(a, p.stats[(size_t)b * S + s], p.k2);
    }
    const int x = p.x_b[b];
    int k = -1;
    if (bad || !(a.m > -1.0e38f) || nb == 0) {
      status_or(p.dev_status, SD_DEV_NONFINITE);
    } else if (x < 0 || x >= p.V) {
      status_or(p.dev_status, SD_DEV_BAD_TOKEN);
    } else {
      float qx;
      if (p.greedy) {
        qx = x == key_idx(best[0]) ? 1.f : 0.f;
      } else {
        const char *row = static_cast<const char *>(p.draft) +
                          (size_t)b * p.V * (p.dt == SD_F32 ? 4 : 2);
        const float zx = p.dt == SD_F32 ? load_logit<0>(row, x)
                                        : load_logit<1>(row, x);
        qx = ex2((zx - a.m) * p.k2) / a.s;
      }
      // floor(k_max (1 - q)) = k_max - ceil(k_max q), exact for tiny q
      k = F - (int)ceilf((float)F * qx);
      k = max(1, min(k, p.V));
    }
    k_s = k;
    p.out_k[b] = k;
  }
  __syncthreads();
  const int k = k_s;
  for (int i = tid; i < F; i += kThreads)
    p.out_tokens[(size_t)b * F + i] = i < k ? key_idx(best[i]) : -1;
}

}  // namespace sdv

namespace {

using namespace sdv;

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Slices per row: enough CTAs for ~4 per SM, slices of >= 256 vectors, and
// slices x keys within what the merge ranks in shared memory.
int slice_bound(long long nvec, int F) {
  long long s = nvec / 256;
  if (s < 1) s = 1;
  const long long cap = kPrestoMaxKeys / F;
  return (int)(s < cap ? s : cap);
}

// Resident CTAs per SM of a kernel at kThreads threads (cached).
int resident_per_sm(const void *kern) {
  static std::mutex mu;
  static std::unordered_map<const void *, int> cache;
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(kern);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, 0) !=
          cudaSuccess ||
      n < 1)
    n = 1;
  cache[kern] = n;
  return n;
}

// As many slices as one full wave of CTAs allows (no partial wave), within
// the bound above.
int choose_slices(long long nvec, long long items, int F, int sms,
                  const void *kern) {
  const int bound = slice_bound(nvec, F);
  long long s = (long long)resident_per_sm(kern) * sms / items;
  if (s < 1) s = 1;
  return (int)(s < bound ? s : bound);
}

struct SelWs {
  uint64_t *keys;
  MS *stats;
  int *bad;
};

size_t sel_ws_bytes(long long items, int S, int F) {
  return align256((size_t)items * S * F * 8) + align256((size_t)items * S * 8) +
         align256((size_t)items * S * 4);
}

SelWs sel_ws(void *ws, long long items, int S, int F) {
  char *c = static_cast<char *>(ws);
  SelWs w;
  w.keys = reinterpret_cast<uint64_t *>(c);
  c += align256((size_t)items * S * F * 8);
  w.stats = reinterpret_cast<MS *>(c);
  c += align256((size_t)items * S * 8);
  w.bad = reinterpret_cast<int *>(c);
  return w;
}

using SelKernel = void (*)(const SelParams);

SelKernel pick_sel(sd_dtype dt, bool vec, bool rho) {
  if (dt == SD_F32) {
    if (vec)
      return rho ? presto_select_kernel<0, 4, true>
                 : presto_select_kernel<0, 4, false>;
    return rho ? presto_select_kernel<0, 1, true>
               : presto_select_kernel<0, 1, false>;
  }
  if (vec)
    return rho ? presto_select_kernel<1, 8, true>
               : presto_select_kernel<1, 8, false>;
  return rho ? presto_select_kernel<1, 1, true>
             : presto_select_kernel<1, 1, false>;
}

__global__ void presto_init_kernel(int B, int W, int budget,
                                   int32_t *n_nodes, int32_t *parent,
                                   int32_t *node_tokens, float *node_score,
                                   int32_t *frontier_node,
                                   float *frontier_score) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long nn = (long long)B * budget, nf = (long long)B * W;
  if (i < nn) {
    parent[i] = -1;
    node_tokens[i] = -1;
    node_score[i] = 0.f;
  }
  if (i < nf) {
    frontier_node[i] = (i % W) == 0 ? 0 : -1;
    frontier_score[i] = 0.f;
  }
  if (i < B) n_nodes[i] = 1;
}

}  // namespace

extern "C" sd_status sd_presto_init(int B, int W, int budget,
                                    int32_t *n_nodes, int32_t *parent,
                                    int32_t *node_tokens, float *node_score,
                                    int32_t *frontier_node,
                                    float *frontier_score, void *stream) {
  SDV_REQUIRE(B >= 0, "B < 0");
  SDV_REQUIRE(W >= 1 && W <= SD_MAX_FANOUT, "W=%d outside [1, %d]", W,
              SD_MAX_FANOUT);
  SDV_REQUIRE(budget >= 1, "budget < 1");
  if (B == 0) return SD_OK;
  SDV_REQUIRE(n_nodes && parent && node_tokens && node_score &&
                  frontier_node && frontier_score,
              "null pointer");
  int sms = 0;
  sd_status st = check_device(&sms);
  if (st != SD_OK) return st;
  long long n = (long long)B * (budget > W ? budget : W);
  const int threads = 256;
  const long long blocks = (n + threads - 1) / threads;
  presto_init_kernel<<<(unsigned)blocks, threads, 0,
                       static_cast<cudaStream_t>(stream)>>>(
      B, W, budget, n_nodes, parent, node_tokens, node_score, frontier_node,
      frontier_score);
  SDV_CUDA(cudaGetLastError());
  return SD_OK;
}

extern "C" size_t sd_presto_expand_workspace(int B, int W, int V, int b_top,
                                             sd_dtype dt) {
  (void)dt;
  if (B < 0 || W < 1 || V < 1 || b_top < 1 || b_top > SD_MAX_FANOUT)
    return 256;
  const long long items = (long long)B * W;
  return sel_ws_bytes(items, slice_bound(V, b_top), b_top);
}

extern "C" sd_status sd_presto_expand(
    const void *q_logits, long long q_stride, const void *log_rho,
    sd_dtype dt, int B, int W, int V, float T, float lambda, int b_top,
    int budget, int32_t *n_nodes, int32_t *parent, int32_t *node_tokens,
    float *node_score, int32_t *frontier_node, float *frontier_score,
    int32_t *dev_status, void *workspace, size_t ws_bytes, void *stream) {
  SDV_REQUIRE(dt == SD_F32 || dt == SD_BF16, "bad dtype %d", (int)dt);
  SDV_REQUIRE(B >= 0, "B < 0");
  SDV_REQUIRE(W >= 1 && W <= SD_MAX_FANOUT, "W=%d outside [1, %d]", W,
              SD_MAX_FANOUT);
  SDV_REQUIRE(V >= 1 && V <= SD_MAX_V, "V=%d outside [1, %d]", V, SD_MAX_V);
  SDV_REQUIRE(b_top >= 1 && b_top <= SD_MAX_FANOUT,
              "b_top=%d outside [1, %d]", b_top, SD_MAX_FANOUT);
  if ((long long)W * b_top > kPrestoMaxCand)
    return fail(SD_ERR_UNSUPPORTED, "W b_top = %d above %d", W * b_top,
                kPrestoMaxCand);
  SDV_REQUIRE(budget >= 1, "budget < 1");
  SDV_REQUIRE(T > 0.f && std::isfinite(T), "T must be finite and > 0");
  SDV_REQUIRE(lambda >= 0.f && std::isfinite(lambda),
              "lambda must be finite and >= 0");
  SDV_REQUIRE(q_stride >= V, "q_stride < V");
  if (B == 0) return SD_OK;
  SDV_REQUIRE(q_logits && (lambda == 0.f || log_rho) && n_nodes && parent &&
                  node_tokens && node_score && frontier_node &&
                  frontier_score,
              "null pointer");
  int sms = 0;
  sd_status st = check_device(&sms);
  if (st != SD_OK) return st;
  const int eb = dt == SD_F32 ? 4 : 2, vw = dt == SD_F32 ? 4 : 8;
  const bool rho = lambda != 0.f;
  const bool vec = aligned16(q_logits) && (q_stride * eb) % 16 == 0 &&
                   ((size_t)V * eb) % 16 == 0 && (!rho || aligned16(log_rho));
  const long long nvec = vec ? V / vw : V;
  const long long items = (long long)B * W;
  const SelKernel kern = pick_sel(dt, vec, rho);
  const int S = choose_slices(nvec, items, b_top, sms, (const void *)kern);
  const size_t need = sel_ws_bytes(items, S, b_top);
  if (!workspace || ws_bytes < need)
    return fail(SD_ERR_INVALID_ARG, "workspace of >= %zu bytes required",
                need);
  const SelWs w = sel_ws(workspace, items, S, b_top);
  SelParams sp;
  sp.q = q_logits;
  sp.q_stride = q_stride;
  sp.rho = log_rho;
  sp.B = B;
  sp.W = W;
  sp.V = V;
  sp.S = S;
  sp.scale = 1.f / T;
  sp.lambda = lambda;
  sp.k2 = (float)(1.4426950408889634 / (double)T);
  sp.F = b_top;
  sp.frontier_node = frontier_node;
  sp.n_nodes = n_nodes;
  sp.budget = budget;
  sp.keys = w.keys;
  sp.stats = w.stats;
  sp.bad = w.bad;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  {
    void *args[] = {&sp};
    const sd_status st2 =
        launch_pdl((const void *)kern, (unsigned)(items * S), kThreads, 0, s,
                   args);
    if (st2 != SD_OK) return st2;
  }
  MergeParams mp;
  mp.keys = w.keys;
  mp.stats = w.stats;
  mp.bad = w.bad;
  mp.B = B;
  mp.W = W;
  mp.S = S;
  mp.F = b_top;
  mp.k2 = sp.k2;
  mp.scale = sp.scale;
  mp.budget = budget;
  mp.n_nodes = n_nodes;
  mp.parent = parent;
  mp.node_tokens = node_tokens;
  mp.node_score = node_score;
  mp.frontier_node = frontier_node;
  mp.frontier_score = frontier_score;
  mp.dev_status = dev_status;
  void *margs[] = {&mp};
  return launch_pdl((const void *)presto_merge_kernel, (unsigned)B, kThreads,
                    0, s, margs);
}

extern "C" size_t sd_branch_fork_workspace(int B, int V, int k_max,
                                           sd_dtype dt) {
  (void)dt;
  if (B < 0 || V < 1 || k_max < 1 || k_max > SD_MAX_FANOUT) return 256;
  return sel_ws_bytes(B, slice_bound(V, k_max), k_max);
}

extern "C" sd_status sd_branch_fork(const void *draft_logits, sd_dtype dt,
                                    const int32_t *x_b, int B, int V, float T,
                                    int k_max, int32_t *out_k,
                                    int32_t *out_tokens, int32_t *dev_status,
                                    void *workspace, size_t ws_bytes,
                                    void *stream) {
  SDV_REQUIRE(dt == SD_F32 || dt == SD_BF16, "bad dtype %d", (int)dt);
  SDV_REQUIRE(B >= 0, "B < 0");
  SDV_REQUIRE(V >= 1 && V <= SD_MAX_V, "V=%d outside [1, %d]", V, SD_MAX_V);
  SDV_REQUIRE(k_max >= 1 && k_max <= SD_MAX_FANOUT,
              "k_max=%d outside [1, %d]", k_max, SD_MAX_FANOUT);
  SDV_REQUIRE(T >= 0.f && std::isfinite(T), "T must be finite and >= 0");
  if (B == 0) return SD_OK;
  SDV_REQUIRE(draft_logits && x_b && out_k && out_tokens, "null pointer");
  int sms = 0;
  sd_status st = check_device(&sms);
  if (st != SD_OK) return st;
  const int eb = dt == SD_F32 ? 4 : 2, vw = dt == SD_F32 ? 4 : 8;
  const bool vec = aligned16(draft_logits) && ((size_t)V * eb) % 16 == 0;
  const long long nvec = vec ? V / vw : V;
  const SelKernel kern = pick_sel(dt, vec, false);
  const int S = choose_slices(nvec, B, k_max, sms, (const void *)kern);
  const size_t need = sel_ws_bytes(B, S, k_max);
  if (!workspace || ws_bytes < need)
    return fail(SD_ERR_INVALID_ARG, "workspace of >= %zu bytes required",
                need);
  const SelWs w = sel_ws(workspace, B, S, k_max);
  SelParams sp;
  sp.q = draft_logits;
  sp.q_stride = V;
  sp.rho = nullptr;
  sp.B = B;
  sp.W = 1;
  sp.V = V;
  sp.S = S;
  sp.scale = 1.f;  // ordered by the logits themselves
  sp.lambda = 0.f;
  sp.k2 = T > 0.f ? (float)(1.4426950408889634 / (double)T) : 0.f;
  sp.F = k_max;
  sp.frontier_node = nullptr;
  sp.n_nodes = nullptr;
  sp.budget = 1;
  sp.keys = w.keys;
  sp.stats = w.stats;
  sp.bad = w.bad;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  {
    void *args[] = {&sp};
    const sd_status st2 = launch_pdl((const void *)kern,
                                     (unsigned)((long long)B * S), kThreads,
                                     0, s, args);
    if (st2 != SD_OK) return st2;
  }
  ForkParams fp;
  fp.keys = w.keys;
  fp.stats = w.stats;
  fp.bad = w.bad;
  fp.draft = draft_logits;
  fp.dt = (int)dt;
  fp.B = B;
  fp.V = V;
  fp.S = S;
  fp.F = k_max;
  fp.k2 = sp.k2;
  fp.greedy = T == 0.f;
  fp.x_b = x_b;
  fp.out_k = out_k;
  fp.out_tokens = out_tokens;
  fp.dev_status = dev_status;
  void *fargs[] = {&fp};
  return launch_pdl((const void *)fork_merge_kernel, (unsigned)B, kThreads, 0,
                    s, fargs);
}
