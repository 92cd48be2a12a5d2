// sdv_allrows.cu -- linear verify ("01 · Draft-then-verify", Algorithm 1)
// for small inputs: every row's statistics at once, then one decision per
// sequence.
//
// The cluster kernel of sdv_linear.cu reads a sequence's rows position by
// position and stops at the first rejection, paying a cluster barrier and
// a decision per position.  When the whole input is a few tens of MB (a
// small batch, or a short vocabulary), that chain of barriers, not HBM, is
// the cost.  Here:
//  1. one launch computes the (max, sum) (or argmax, at T = 0) of every
//     row the scan could need -- target rows 0..gamma and draft rows
//     0..gamma-1 of every sequence -- each row cut into S slices over
//     S CTAs: all rows are read once, at full bandwidth, with no early
//     exit;
//  2. one CTA per sequence merges its rows' slices, gathers the logits at
//     the draft tokens, applies the accept tests in position order, and
//     draws the correction norm(max(0, p_n - q_n)) or the bonus p_gamma by
//     inverse CDF over the two rows of position n (a second read of those
//     two rows only).
// The arithmetic is that of the cluster kernel: the same (max, sum)
// states, the same accept ratio, the same residual weights and draw.
#include "sdv_device.cuh"
#include "sdv_host.cuh"

namespace sdv {

constexpr int kARMaxSlices = 32;  // slices per row (one warp merges them)

struct ARParams {
  const void *target;  // [B, gamma+1, V]
  const void *draft;   // row j of sequence b at b * d_seq_rows + j
  long long d_seq_rows;
  const int32_t *tokens;
  const float *uniforms;
  int B, gamma, V;
  float k2;
  int S;     // slices per row
  int rows;  // rows per sequence: gamma + 1 targets (+ gamma drafts)
  MS *part;  // [B][rows][S]
  AM *apart;
  int32_t *n_acc, *out_tokens;
  float *out_prob, *out_accept;
  int32_t *dev_status;
};

template <int DT>
__device__ __forceinline__ const char *ar_row(const ARParams &p, int b,
                                              int r) {
  const size_t rowb = (size_t)p.V * elt_bytes<DT>();
  if (r <= p.gamma)
    return static_cast<const char *>(p.target) +
           ((size_t)b * (p.gamma + 1) + r) * rowb;
  return static_cast<const char *>(p.draft) +
         ((size_t)b * p.d_seq_rows + (r - p.gamma - 1)) * rowb;
}

template <int DT, int VW, bool GREEDY>
__global__ void __launch_bounds__(kThreads)
    allrows_stats_kernel(const ARParams p) {
  __shared__ MS red[1][kWarps];
  __shared__ AM ared[kWarps];
  const int s = blockIdx.x % p.S;
  const int rr = blockIdx.x / p.S;  // row over the batch
  const int b = rr / p.rows, r = rr % p.rows;
  const GRow<DT, VW> row{ar_row<DT>(p, b, r)};
  const Slice sl = make_slice(p.V / VW, s, p.S);
  if constexpr (GREEDY) {
    AM a = am_empty();
    argmax_pass<DT, VW>(row, sl, a);
    a = block_reduce_am(a, ared);
    if (threadIdx.x == 0) p.apart[(size_t)rr * p.S + s] = a;
  } else {
    MS st[1] = {ms_empty()};
    MS unused = ms_empty();
    stats_pass<DT, VW>(row, row, false, sl, p.k2, st[0], unused);
    block_reduce_ms<1>(st, p.k2, red);
    if (threadIdx.x == 0) p.part[(size_t)rr * p.S + s] = st[0];
  }
}

struct ARSmem {
  MS mrg[2 * SD_MAX_GAMMA + 1];
  AM amrg[SD_MAX_GAMMA + 1];
  int gx[SD_MAX_GAMMA];
  float gzt[SD_MAX_GAMMA], gzd[SD_MAX_GAMMA], gr[SD_MAX_GAMMA];
  int n, kind, bad, tok;
  MS mt, md;
  DrawSmem draw;
};

// One cluster per sequence: every CTA makes the same decision, and the
// draw's pass over the two rows of position n is cut into one slice per
// CTA (cluster_draw).
template <int DT, int VW, bool GREEDY>
__global__ void __launch_bounds__(kThreads)
    allrows_decide_kernel(const ARParams p) {
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ ARSmem sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rank = (int)cluster.block_rank(), CL = (int)cluster.num_blocks();
  const int b = (int)(blockIdx.x / CL);
  const int gamma = p.gamma, G1 = gamma + 1, V = p.V;
  const float k2 = p.k2;
  float *segmass = reinterpret_cast<float *>(dsm);
  // merge each row's slice states (rows: targets 0..gamma, drafts after)
  for (int r = warp; r < p.rows; r += kWarps) {
    const size_t base = ((size_t)b * p.rows + r) * p.S;
    if constexpr (GREEDY) {
      AM a = lane < p.S ? p.apart[base + lane] : am_empty();
      a = warp_down_am(a);
      if (lane == 0) sh.amrg[r] = a;
    } else {
      MS m = lane < p.S ? p.part[base + lane] : ms_empty();
      m = warp_down_ms(m, k2);
      if (lane == 0) sh.mrg[r] = m;
    }
  }
  // the draft tokens, their logits and the accept uniforms
  for (int j = tid; j < gamma; j += kThreads) {
    const int x = p.tokens[(size_t)b * gamma + j];
    float zt = 0.f, zd = 0.f, r = 0.f;
    if (!GREEDY && x >= 0 && x < V) {
      zt = load_logit<DT>(ar_row<DT>(p, b, j), x);
      zd = load_logit<DT>(ar_row<DT>(p, b, G1 + j), x);
    }
    if (!GREEDY) r = p.uniforms[(size_t)b * G1 + j];
    sh.gx[j] = x;
    sh.gzt[j] = zt;
    sh.gzd[j] = zd;
    sh.gr[j] = r;
  }
  __syncthreads();
  if (tid == 0) {  // the accept tests in position order
    int n = 0, kind = 0, bad_any = 0, tok = -1;
    MS mt = ms_empty(), md = ms_empty();
    for (int j = 0; j <= gamma && !kind; ++j) {
      const int x = j < gamma ? sh.gx[j] : 0;
      const bool bad = j < gamma && (x < 0 || x >= V);
      bad_any |= bad;
      bool invalid, acc = false;
      float accp = 0.f;
      if constexpr (GREEDY) {
        const AM a = sh.amrg[j];
        invalid = a.bad || !(a.v > -kInf);
        acc = !invalid && j < gamma && x == a.i;
        accp = acc ? 1.f : 0.f;
        tok = a.i;
      } else {
        mt = sh.mrg[j];
        md = j < gamma ? sh.mrg[G1 + j] : ms_empty();
        invalid = !ms_valid(mt) || (j < gamma && !ms_valid(md));
        if (!invalid && j < gamma && !bad) {
          const float rho = accept_ratio(sh.gzt[j], sh.gzd[j], mt, md, k2);
          acc = sh.gr[j] <= rho;
          accp = fminf(1.f, rho);
        }
      }
      if (rank == 0 && p.out_accept && j < gamma && !invalid)
        p.out_accept[(size_t)b * gamma + j] = accp;
      if (invalid) kind = 3;
      else if (j == gamma) kind = 2;
      else if (!acc) kind = 1;
      else ++n;
    }
    sh.n = n;
    sh.kind = kind;
    sh.bad = bad_any;
    sh.tok = tok;
    sh.mt = mt;
    sh.md = md;
  }
  __syncthreads();
  const int n = sh.n, kind = sh.kind, bad_token = sh.bad;
  if (kind == 3) {  // unusable row: outputs -1
    if (rank != 0) return;
    for (int t = tid; t <= gamma; t += kThreads)
      p.out_tokens[(size_t)b * G1 + t] = -1;
    if (p.out_accept)
      for (int t = n + tid; t < gamma; t += kThreads)
        p.out_accept[(size_t)b * gamma + t] = -1.f;
    if (tid == 0) {
      p.n_acc[b] = -1;
      if (p.out_prob) p.out_prob[b] = 0.f;
      status_or(p.dev_status,
                SD_DEV_NONFINITE | (bad_token ? SD_DEV_BAD_TOKEN : 0));
    }
    return;
  }
  int tok = sh.tok, zero_mass = 0;
  float prob = 1.f;
  if constexpr (!GREEDY) {
    // correction (kind 1) or bonus (kind 2) by inverse CDF over the rows of
    // position n
    const GRow<DT, VW> ra{ar_row<DT>(p, b, n)};
    const GRow<DT, VW> rb{kind == 1 ? ar_row<DT>(p, b, G1 + n)
                                    : ar_row<DT>(p, b, n)};
    bool has_q = kind == 1;
    Weight W;
    W.k2 = k2;
    W.mtk = sh.mt.m * k2;
    W.ist = 1.f / sh.mt.s;
    W.mdk = sh.md.m * k2;
    W.cq = 1.f / sh.md.s;
    const float u = p.uniforms[(size_t)b * G1 + gamma];
    const Slice sl = make_slice(V / VW, rank, CL);
    int par = 0;
    DrawOut o;
    for (int attempt = 0; attempt < 2; ++attempt) {
      o = cluster_draw<DT, VW>(cluster, sh.draw, segmass, ra, rb, has_q, W,
                               sl, u, par);
      if (o.owner >= 0) break;
      zero_mass = 1;  // residual of zero mass: draw from p_n instead
      has_q = false;
      __syncthreads();
    }
    // no CTA leaves while a peer may still read its shared memory
    cluster.sync();
    if (o.owner != rank || warp != 0) return;  // it holds the drawn token
    tok = o.t;
    prob = (float)((double)o.wt / o.N);
  } else {
    if (rank != 0 || warp != 0) return;
  }
  for (int t = lane; t <= gamma; t += 32) {
    int v = -1;
    if (t < n) v = p.tokens[(size_t)b * gamma + t];
    else if (t == n) v = tok;
    p.out_tokens[(size_t)b * G1 + t] = v;
  }
  if (p.out_accept)
    for (int t = n + 1 + lane; t < gamma; t += 32)
      p.out_accept[(size_t)b * gamma + t] = -1.f;
  if (lane == 0) {
    p.n_acc[b] = n;
    if (p.out_prob) p.out_prob[b] = prob;
    status_or(p.dev_status, (bad_token ? SD_DEV_BAD_TOKEN : 0) |
                                (zero_mass ? SD_DEV_ZERO_MASS : 0));
  }
}

}  // namespace sdv

namespace sdv {

namespace {

constexpr long long kARMaxBytes = 64ll << 20;  // rows read by the path
constexpr size_t kARMaxWs = 512 << 10;         // its slice states
constexpr long long kARMaxVecs = 48 * 1024 / 4 * 32;  // segments in smem

long long ar_nvec(int V, sd_dtype dt, bool vec) {
  return vec ? V / (dt == SD_F32 ? 4 : 8) : V;
}

int ar_smax(long long nvec) {
  long long s = nvec / 256;
  if (s < 1) s = 1;
  return (int)(s < kARMaxSlices ? s : kARMaxSlices);
}

size_t ar_ws_bytes(int B, int rows, int S) {
  return ((size_t)B * rows * S * sizeof(AM) + 255) / 256 * 256;
}

using ARKernel = void (*)(const ARParams);

template <int DT, int VW>
void ar_pick(bool greedy, ARKernel *stats, ARKernel *decide) {
  *stats = greedy ? allrows_stats_kernel<DT, VW, true>
                  : allrows_stats_kernel<DT, VW, false>;
  *decide = greedy ? allrows_decide_kernel<DT, VW, true>
                   : allrows_decide_kernel<DT, VW, false>;
}

}  // namespace

// Bytes of workspace the path may need at these sizes under any setting of
// SD_TUNE_ALLROWS (0 when it can never be taken); sampling rows assumed.
// The path is chosen from the sizes and that switch alone, never from how
// much scratch a caller hands over beyond this figure, so every entry that
// sizes its scratch by the query takes the same path.
size_t allrows_workspace(int B, int gamma, int V, sd_dtype dt) {
  (void)dt;
  if (B <= 0 || V <= 0 || gamma < 0) return 0;
  const int rows = 2 * gamma + 1;
  const size_t w = ar_ws_bytes(B, rows, ar_smax(V));  // V >= nvec
  return w <= kARMaxWs ? w : 0;
}

// Whether the all-rows path takes this call: small inputs (SD_TUNE_ALLROWS 0
// never, 2 whenever it fits), no residual output, workspace enough.
bool use_allrows(int B, int gamma, int V, sd_dtype dt, const void *target,
                 const void *draft, float T, const float *out_resid,
                 size_t ws_bytes) {
  const int mode = tune(SD_TUNE_ALLROWS);
  if (mode == 0 || out_resid || B <= 0) return false;
  const int eb = dt == SD_F32 ? 4 : 2;
  const bool greedy = T == 0.f;
  const bool vec = aligned16(target) && (greedy || gamma == 0 ||
                                         aligned16(draft)) &&
                   ((size_t)V * eb) % 16 == 0;
  const long long nvec = ar_nvec(V, dt, vec);
  const int rows = gamma + 1 + (greedy ? 0 : gamma);
  if (nvec > kARMaxVecs) return false;
  const size_t need = ar_ws_bytes(B, rows, ar_smax(nvec));
  const size_t query = allrows_workspace(B, gamma, V, dt);  // >= need if > 0
  if (query == 0 || need > query || need > ws_bytes) return false;
  return mode == 2 || (long long)B * rows * V * eb <= kARMaxBytes;
}

sd_status allrows_launch(const void *target, const void *draft, sd_dtype dt,
                         long long d_seq_rows, const int32_t *tokens,
                         const float *uniforms, int B, int gamma, int V,
                         float T, int32_t *n_acc, int32_t *out_tokens,
                         float *out_prob, float *out_accept,
                         int32_t *dev_status, void *ws, size_t ws_bytes,
                         cudaStream_t stream) {
  int sms = 0;
  sd_status st = check_device(&sms);
  if (st != SD_OK) return st;
  const bool greedy = T == 0.f;
  const int eb = dt == SD_F32 ? 4 : 2;
  const bool vec = aligned16(target) && (greedy || gamma == 0 ||
                                         aligned16(draft)) &&
                   ((size_t)V * eb) % 16 == 0;
  const long long nvec = ar_nvec(V, dt, vec);
  const int rows = gamma + 1 + (greedy ? 0 : gamma);
  // slices: about four CTAs per SM over all rows, slices of >= 256 vectors
  long long S = (4LL * sms + (long long)B * rows - 1) / ((long long)B * rows);
  if (S < 1) S = 1;
  if (S > ar_smax(nvec)) S = ar_smax(nvec);
  if (!ws || ws_bytes < ar_ws_bytes(B, rows, (int)S))
    return fail(SD_ERR_INVALID_ARG, "workspace too small");
  ARParams prm;
  prm.target = target;
  prm.draft = draft;
  prm.d_seq_rows = d_seq_rows;
  prm.tokens = tokens;
  prm.uniforms = uniforms;
  prm.B = B;
  prm.gamma = gamma;
  prm.V = V;
  prm.k2 = greedy ? 0.f : (float)(1.4426950408889634 / (double)T);
  prm.S = (int)S;
  prm.rows = rows;
  prm.part = static_cast<MS *>(ws);
  prm.apart = static_cast<AM *>(ws);
  prm.n_acc = n_acc;
  prm.out_tokens = out_tokens;
  prm.out_prob = out_prob;
  prm.out_accept = out_accept;
  prm.dev_status = dev_status;
  ARKernel stats = nullptr, decide = nullptr;
  if (dt == SD_F32) {
    if (vec) ar_pick<0, 4>(greedy, &stats, &decide);
    else ar_pick<0, 1>(greedy, &stats, &decide);
  } else {
    if (vec) ar_pick<1, 8>(greedy, &stats, &decide);
    else ar_pick<1, 1>(greedy, &stats, &decide);
  }
  stats<<<(unsigned)((long long)B * rows * S), kThreads, 0, stream>>>(prm);
  SDV_CUDA(cudaGetLastError());
  // the decision's cluster: the draw's slices of at least ~512 vectors
  int CLd = 1;
  while (CLd < 8 && nvec / (2 * CLd) >= 512) CLd *= 2;
  const long long per = (nvec + CLd - 1) / CLd;
  const size_t smem = ((size_t)((per + 31) / 32) * 4 + 127) / 128 * 128;
  void *args[] = {&prm};
  return launch_clusters((const void *)decide, B, CLd, smem, stream, args);
}

}  // namespace sdv
