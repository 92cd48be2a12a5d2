// sdv_fanout.cu -- top-F_k draft tokens per lookahead position (Speculative
// Speculative Decoding / Saguaro, "speculation cache strategy": the cache
// is filled with the top-F_k tokens of the draft logits at each lookahead
// position k; F follows the geometric fan-out of Theorem 12).
//
// One cluster (usually a single CTA) owns one row at a time; rows all have
// the same cost, so clusters take them round-robin.  Each CTA streams its
// slice once through the TMA ring (16-byte aligned rows; SD_TUNE_FANOUT_LDG
// takes 16-byte loads instead) or with scalar loads, filtering it through
// per-warp sorted lists against a CTA-wide threshold (sdv_topf.cuh); the
// warps' lists are ranked together, and for clusters of several CTAs rank 0
// merges the slice lists read through distributed shared memory.
#include "sdv_host.cuh"
#include "sdv_fanrow.cuh"

namespace sdv {

struct FanParams {
  const void *draft;  // [B, K+1, V]
  int B, K, V;
  int F[SD_MAX_K + 1];
  int off[SD_MAX_K + 2];
  int32_t *out_tokens;  // [B, total]
  float *out_logit;
  int32_t *dev_status;
  int nclusters;
  int seg_bytes;
  int evict_first;  // read the rows with an L2 evict-first policy
};

struct FanSmem {
  TopSmem top;
  uint64_t slot[2][SD_MAX_FANOUT];  // [parity] this CTA's list (peers read)
  int slot_n[2];
  int slot_nan[2];
  int nan_flag;
};

constexpr int kUF = 8;  // vectors in flight per thread on the load path

// Stream one row slice through the warp filters with 16-byte loads; warp w
// takes the blocks of 32 * kUF vectors w, w + kWarps, ...
template <int DT, int VW>
__device__ __forceinline__ void filter_pass(const char *row, const Slice &sl,
                                            WarpFilter &w, uint32_t *cta_th) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int vb = sl.vbeg + warp * 32 * kUF; vb < sl.vend;
       vb += kWarps * 32 * kUF) {  // warp-uniform
    Raw<DT, VW> x[kUF];
#pragma unroll
    for (int u = 0; u < kUF; ++u) {
      const int v = vb + u * 32 + lane;
      if (v < sl.vend) x[u] = load_vec<DT, VW>(row, v);
    }
    wf_sync(w, cta_th);
#pragma unroll
    for (int u = 0; u < kUF; ++u) {
      const int v = vb + u * 32 + lane;
      wf_offer<DT, VW>(w, cta_th, x[u], v < sl.vend, v * VW);
    }
  }
}

// Select the exact top-F of a row over a cluster and (rank 0) write it.
template <int DT, int VW, bool RING>
__device__ void row_topf(cg::cluster_group &cluster, FanSmem &sh, Ring &rg,
                         const char *row, const Slice &sl, int F,
                         int32_t *otok, float *olog, int32_t *dev_status,
                         int &par) {
  const int tid = threadIdx.x;
  const int rank = (int)cluster.block_rank(), CL = (int)cluster.num_blocks();
  WarpFilter w;
  wf_init(w, F);
  if constexpr (RING) filter_pass_ring<DT, VW>(rg, row, sl, w, &sh.top.th);
  else filter_pass<DT, VW>(row, sl, w, &sh.top.th);
  const int anynan = __syncthreads_or(w.nseen != w.nseen);
  wf_export(w, sh.top);
  __syncthreads();
  const int nout = rank_select(sh.top, kWarps * F, F);
  if (tid == 0) sh.top.th = 0;  // every warp has finished filtering
  if (CL == 1) {
    for (int i = tid; i < F; i += kThreads) {
      const bool ok = !anynan && i < nout;
      otok[i] = ok ? key_idx(sh.top.out[i]) : -1;
      if (olog) olog[i] = ok ? key_val(sh.top.out[i]) : __int_as_float(0x7fc00000);
    }
    if (tid == 0 && anynan) status_or(dev_status, SD_DEV_NONFINITE);
    __syncthreads();
    return;
  }
  for (int i = tid; i < F; i += kThreads)
    sh.slot[par][i] = i < nout ? sh.top.out[i] : 0;
  if (tid == 0) {
    sh.slot_n[par] = nout;
    sh.slot_nan[par] = anynan;
  }
  cluster.sync();
  if (rank == 0) {
    // gather the CL lists (CL * F <= kWarps * SD_MAX_FANOUT) and rank them
    int C = 0;
    if (tid == 0) sh.nan_flag = 0;
    __syncthreads();
    for (int r = 0; r < CL; ++r) {
      const FanSmem *rs = cluster.map_shared_rank(&sh, r);
      const int nr = rs->slot_n[par];
      for (int i = tid; i < nr; i += kThreads) sh.top.flat[C + i] = rs->slot[par][i];
      if (tid == 0 && rs->slot_nan[par]) sh.nan_flag = 1;
      C += nr;
    }
    __syncthreads();
    const int n = rank_select(sh.top, C, F);
    const int bad = sh.nan_flag;
    for (int i = tid; i < F; i += kThreads) {
      const bool ok = !bad && i < n;
      otok[i] = ok ? key_idx(sh.top.out[i]) : -1;
      if (olog) olog[i] = ok ? key_val(sh.top.out[i]) : __int_as_float(0x7fc00000);
    }
    if (tid == 0 && bad) status_or(dev_status, SD_DEV_NONFINITE);
  }
  par ^= 1;
  __syncthreads();
}

#ifndef SDV_FAN_MINB
#define SDV_FAN_MINB 4
#endif

template <int DT, int VW, bool RING>
__global__ void __launch_bounds__(kThreads, SDV_FAN_MINB)
    fanout_kernel(const FanParams p) {
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ FanSmem sh;
  __shared__ uint64_t bars[2 * kStages];
  Ring rg;
  rg.buf = reinterpret_cast<uint4 *>(dsm + p.seg_bytes);
  rg.full = bars;
  rg.empty = bars + kStages;
  rg.dev_status = p.dev_status;
  if (threadIdx.x == 0) sh.top.th = 0;
  if (RING) {
    ring_init(rg);
    // every row is read once: keep it from pushing out lines that a kernel
    // running beside this one reads again
    if (p.evict_first) rg.policy = l2_evict_first_policy();
  }
  else __syncthreads();
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank(), CL = (int)cluster.num_blocks();
  const int V = p.V, K1 = p.K + 1;
  const Slice sl = make_slice(V / VW, rank, CL);
  const size_t rowb = (size_t)V * elt_bytes<DT>();
  const char *base = static_cast<const char *>(p.draft);
  const int total = p.off[K1];
  int par = 0;
  const long long rows = (long long)p.B * K1;
  for (long long r = blockIdx.x / CL; r < rows; r += p.nclusters) {
    const int b = (int)(r / K1), k = (int)(r % K1);
    const int F = p.F[k];
    if (F == 0) continue;
    int32_t *otok = p.out_tokens + (size_t)b * total + p.off[k];
    float *olog = p.out_logit ? p.out_logit + (size_t)b * total + p.off[k]
                              : nullptr;
    row_topf<DT, VW, RING>(cluster, sh, rg, base + (size_t)r * rowb, sl, F,
                           otok, olog, p.dev_status, par);
  }
  cluster.sync();
}

using FanKernel = void (*)(const FanParams);

static FanKernel pick_fanout(int dt, bool vec, bool ring) {
  if (dt == SD_F32) {
    if (!vec) return fanout_kernel<0, 1, false>;
    return ring ? fanout_kernel<0, 4, true> : fanout_kernel<0, 4, false>;
  }
  if (!vec) return fanout_kernel<1, 1, false>;
  return ring ? fanout_kernel<1, 8, true> : fanout_kernel<1, 8, false>;
}

}  // namespace sdv

extern "C" size_t sd_fanout_topk_workspace(int B, int K, int V, sd_dtype dt) {
  (void)B;
  (void)K;
  (void)V;
  (void)dt;
  return 0;
}

extern "C" sd_status sd_fanout_topk(const void *draft_logits, sd_dtype dt,
                                    int B, int K, int V, const int32_t *F,
                                    int32_t *out_tokens, float *out_logit,
                                    int32_t *dev_status, void *workspace,
                                    size_t ws_bytes, void *stream) {
  using namespace sdv;
  (void)workspace;
  (void)ws_bytes;
  SDV_REQUIRE(dt == SD_F32 || dt == SD_BF16, "bad dtype %d", (int)dt);
  SDV_REQUIRE(B >= 0, "B < 0");
  SDV_REQUIRE(K >= 0 && K <= SD_MAX_K, "K=%d outside [0, %d]", K, SD_MAX_K);
  SDV_REQUIRE(V >= 1 && V <= SD_MAX_V, "V=%d outside [1, %d]", V, SD_MAX_V);
  SDV_REQUIRE(F != nullptr, "F is null");
  FanParams prm;
  int total = 0, maxF = 0;
  for (int k = 0; k <= K; ++k) {
    SDV_REQUIRE(F[k] >= 0, "F[%d] < 0", k);
    if (F[k] > SD_MAX_FANOUT || F[k] > V)
      return fail(SD_ERR_UNSUPPORTED, "F[%d]=%d exceeds min(V, %d)", k, F[k],
                  SD_MAX_FANOUT);
    prm.F[k] = F[k];
    prm.off[k] = total;
    total += F[k];
    maxF = F[k] > maxF ? F[k] : maxF;
  }
  prm.off[K + 1] = total;
  if (B == 0 || total == 0) return SD_OK;
  SDV_REQUIRE(draft_logits && out_tokens, "null pointer");
  int sms = 0;
  sd_status st = check_device(&sms);
  if (st != SD_OK) return st;
  const int eb = dt == SD_F32 ? 4 : 2, vw = dt == SD_F32 ? 4 : 8;
  const bool vec = aligned16(draft_logits) && ((size_t)V * eb) % 16 == 0;
  const long long nvec = V / (vec ? vw : 1);
  const bool ring = vec && tune(SD_TUNE_FANOUT_LDG) == 0;
  FanKernel kern = pick_fanout(dt, vec, ring);
  // rows of equal cost: a single CTA per row unless the rows are too few to
  // fill the GPU, then clusters that split each row
  const long long rows = (long long)B * (K + 1);
  int CL = 1;
  const int forced = tune(SD_TUNE_FANOUT_CLUSTER);
  if (forced == 1 || forced == 2 || forced == 4 || forced == 8 || forced == 16)
    CL = forced;
  else
    while (CL < 16 && rows * CL < 4LL * sms && nvec / (2 * CL) >= 512) CL *= 2;
  // rank 0 gathers the CL lists into kWarps * SD_MAX_FANOUT keys
  while (CL > 1 && CL * maxF > kWarps * SD_MAX_FANOUT) CL /= 2;
  const size_t smem = ring ? 128 + (size_t)kRingBytes : 0;
  int maxc = 0;
  st = max_active_clusters((const void *)kern, CL, smem, &maxc);
  if (st != SD_OK) return st;
  // SD_TUNE_FANOUT_MAXC caps the clusters (tuning: room for a kernel that runs
  // beside this one on another stream)
  const int cap = tune(SD_TUNE_FANOUT_MAXC);
  if (cap > 0 && cap < maxc) maxc = cap;
  // rows of equal cost: give every cluster the same number of them
  const long long per = (rows + maxc - 1) / maxc;
  const long long want = (rows + per - 1) / per;
  prm.draft = draft_logits;
  prm.B = B;
  prm.K = K;
  prm.V = V;
  prm.out_tokens = out_tokens;
  prm.out_logit = out_logit;
  prm.dev_status = dev_status;
  prm.nclusters = (int)want;
  prm.seg_bytes = 128;
  prm.evict_first = tune(SD_TUNE_FANOUT_L2_FIRST) != 0;
  void *args[] = {&prm};
  return launch_clusters((const void *)kern, (int)want, CL, smem,
                         static_cast<cudaStream_t>(stream), args);
}

// ---------------------------------------------------------------- hits
// Saguaro cache hit of each sequence's verification outcome: the speculator
// serves the next round from its cache when the outcome (n accepted, then
// t*) is stored, i.e. when t* is one of the F_n fan-out tokens of position
// n.  One warp per sequence.
namespace sdv {

struct HitParams {
  const int32_t *n_acc;       // [B]
  const int32_t *tokens;      // [B, K+1]
  const int32_t *fan_tokens;  // [B, total]
  int32_t *hit;               // [B]
  int B, K, total;
  int F[SD_MAX_K + 1];
  int off[SD_MAX_K + 2];
};

__global__ void __launch_bounds__(kThreads) fanout_hits_kernel(const HitParams p) {
  const int lane = threadIdx.x & 31;
  const long long b = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (b >= p.B) return;
  const int n = p.n_acc[b];
  if (n < 0 || n > p.K) {
    if (lane == 0) p.hit[b] = -1;
    return;
  }
  const int32_t t = p.tokens[b * (p.K + 1) + n];
  const int32_t *cache = p.fan_tokens + b * p.total + p.off[n];
  bool found = false;
  for (int i = lane; i < p.F[n]; i += 32) found |= cache[i] == t;
  const unsigned any = __ballot_sync(0xffffffffu, found);
  if (lane == 0) p.hit[b] = any ? 1 : 0;
}

}  // namespace sdv

extern "C" sd_status sd_fanout_hits(const int32_t *n_accepted,
                                    const int32_t *out_tokens,
                                    const int32_t *fan_tokens, int B, int K,
                                    const int32_t *F, int32_t *hit,
                                    void *stream) {
  using namespace sdv;
  SDV_REQUIRE(B >= 0, "B < 0");
  SDV_REQUIRE(K >= 0 && K <= SD_MAX_K, "K=%d outside [0, %d]", K, SD_MAX_K);
  SDV_REQUIRE(F != nullptr, "F is null");
  HitParams prm;
  int total = 0;
  for (int k = 0; k <= K; ++k) {
    SDV_REQUIRE(F[k] >= 0, "F[%d] < 0", k);
    prm.F[k] = F[k];
    prm.off[k] = total;
    total += F[k];
  }
  if (B == 0) return SD_OK;
  SDV_REQUIRE(n_accepted && out_tokens && hit, "null pointer");
  SDV_REQUIRE(total == 0 || fan_tokens, "fan_tokens is null");
  int sms = 0;
  sd_status st = check_device(&sms);
  if (st != SD_OK) return st;
  prm.n_acc = n_accepted;
  prm.tokens = out_tokens;
  prm.fan_tokens = fan_tokens;
  prm.hit = hit;
  prm.B = B;
  prm.K = K;
  prm.total = total;
  const int grid = (B + kWarps - 1) / kWarps;
  fanout_hits_kernel<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(prm);
  SDV_CUDA(cudaGetLastError());
  return SD_OK;
}
