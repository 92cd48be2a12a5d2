// sdv_wide.cu -- linear verify for large batches, position by position
// over the whole batch ("01 · Draft-then-verify", Algorithm 1: the accept
// scan is sequential within a sequence, independent across sequences).
//
// Level i is one kernel: every sequence still scanning contributes work
// items (sequence, chunk) -- a chunk of target row i and draft row i --
// spread over all CTAs of the GPU.  Each item streams its chunk through
// the TMA ring, writes the chunk's (max, sum) partials to the workspace and
// bumps the sequence's counter; the CTA that completes a sequence's last
// chunk merges the partials in chunk order and applies the accept test:
// accepted sequences go to level i+1's list, rejected ones (and bonus
// ones at level gamma) to the draw list.  The draws of level i run in
// level i+1's kernel as items of their own (chunk masses of the residual
// max(0, p - q) or of p), and the CTA completing a draw finds the chunk
// that holds u * N and scans it.  No CTA ever waits on another: every
// hand-off is an atomic counter or a kernel boundary, and the kernels are
// chained with programmatic dependent launch.  Only rows up to the first
// rejection are read.
#include "sdv_device.cuh"
#include "sdv_host.cuh"
#include "sdv_ring.cuh"

namespace sdv {

struct SeqState {
  MS mt, md;   // merged stats of the rows of the draw
  int n;       // accepted drafts
  int bad;     // a bad token was seen
};

struct WideWs {
  int *act_n;   // [levels] sequences scanning at each level
  int *act;     // [2][B] their lists (by level parity)
  int *drw_n;   // [levels] draws queued for each level
  int *drw;     // [2][B] entries: seq | (p-only << 30)
  int *cnt;     // [B] items done for the sequence's current stats step
  int *dcnt;    // [B] items done for its draw
  MS *part;     // [B][NC][2]
  double *dmass;  // [B][NC]
  SeqState *st;   // [B]
};

struct WideParams {
  const void *target;
  const void *draft;
  const int32_t *tokens;
  const float *uniforms;
  int B, gamma, V;
  long long d_seq_rows;  // rows per sequence in the draft tensor
  float k2;
  int32_t *n_acc, *out_tokens;
  float *out_prob, *out_accept;
  int32_t *dev_status;
  int level;
  int NC;          // chunks per row
  int chunk_vecs;  // 16-byte vectors per chunk
  int seg_bytes;
  WideWs ws;
};

struct WideSmem {
  MS red[2][kWarps];
  AM ared[kWarps];
  double dred[kWarps];
  int last;
  DrawSmem draw;
};

__device__ __forceinline__ bool last_arrival(int *counter, int total) {
  // every thread's global writes of this item are done (block barrier),
  // made visible device-wide, then one atomic decides who merges
  __shared__ int s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = (atomicAdd(counter, 1) == total - 1);
    if (s_last) __threadfence();
  }
  __syncthreads();
  return s_last != 0;
}

template <int DT, int VW, bool GREEDY>
__global__ void __launch_bounds__(kThreads, 4) wide_level_kernel(const WideParams p) {
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ WideSmem sh;
  __shared__ uint64_t bars[2 * kStages];
  float *segmass = reinterpret_cast<float *>(dsm);
  Ring rg;
  rg.buf = reinterpret_cast<uint4 *>(dsm + p.seg_bytes);
  rg.full = bars;
  rg.empty = bars + kStages;
  rg.dev_status = p.dev_status;
  ring_init(rg);
#if defined(__CUDA_ARCH__)
  // the next level may be scheduled as this grid's CTAs retire; it waits
  // for this grid's completion (and its writes) before reading anything
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i = p.level, gamma = p.gamma, V = p.V, NC = p.NC;
  const int nvec = V / VW;
  const size_t rowb = (size_t)V * elt_bytes<DT>();
  const char *tbase = static_cast<const char *>(p.target);
  const char *dbase = static_cast<const char *>(p.draft);
  const float k2 = p.k2;
  const WideWs &w = p.ws;
  const int A = (i <= gamma) ? (i == 0 ? p.B : w.act_n[i]) : 0;
  const int D = GREEDY ? 0 : w.drw_n[i];
  const long long items = (long long)(A + D) * NC;
  auto chunk_slice = [&](int c) {
    Slice s;
    s.vbeg = c * p.chunk_vecs;
    s.vend = min(nvec, s.vbeg + p.chunk_vecs);
    s.nseg = (s.vend - s.vbeg + 31) >> 5;
    return s;
  };
  auto finish = [&](int s, int n, int t, float prob, int bits, int from) {
    // outputs of a finished sequence (one thread); accept probabilities of
    // positions from .. gamma-1 were never tested
    p.n_acc[s] = n;
    for (int j = 0; j <= gamma; ++j) {
      int v = -1;
      if (n >= 0) {
        if (j < n) v = p.tokens[(size_t)s * gamma + j];
        else if (j == n) v = t;
      }
      p.out_tokens[(size_t)s * (gamma + 1) + j] = v;
    }
    if (p.out_accept)
      for (int j = from; j < gamma; ++j) p.out_accept[(size_t)s * gamma + j] = -1.f;
    if (p.out_prob) p.out_prob[s] = n < 0 ? 0.f : prob;
    status_or(p.dev_status, bits);
  };

  for (long long it = blockIdx.x; it < items; it += gridDim.x) {
    const int idx = (int)(it / NC), c = (int)(it % NC);
    const Slice cs = chunk_slice(c);
    if (idx < A) {
      // ---------------- stats item: chunk c of the rows of position i ----
      const int s = (i == 0) ? idx : w.act[(i & 1) * p.B + idx];
      const bool has_d = !GREEDY && i < gamma;
      const char *trow = tbase + ((size_t)s * (gamma + 1) + i) * rowb;
      const char *drow =
          has_d ? dbase + ((size_t)s * p.d_seq_rows + i) * rowb : nullptr;
      MS *pp = w.part + ((size_t)s * NC + c) * 2;
      if constexpr (GREEDY) {
        AM a = am_empty();
        ring_argmax<DT, VW>(rg, trow, cs, a);
        a = block_reduce_am(a, sh.ared);
        if (tid == 0) {  // an AM stored in the MS slots (same 8+ bytes)
          reinterpret_cast<float *>(pp)[0] = a.v;
          reinterpret_cast<int *>(pp)[1] = a.i;
          reinterpret_cast<int *>(pp)[2] = a.bad;
        }
      } else {
        MS st[2] = {ms_empty(), ms_empty()};
        ring_stats<DT, VW>(rg, trow, drow, cs, k2, st[0], st[1]);
        block_reduce_ms<2>(st, k2, sh.red);
        if (tid == 0) {
          pp[0] = st[0];
          pp[1] = st[1];
        }
      }
      if (!last_arrival(&w.cnt[s], NC)) continue;
      // ---- this CTA completes the sequence's position i: merge, decide ----
      if (warp == 0) {
        // lane l merges chunks l, l+32, ... in order, then a fixed shuffle
        // tree: the same result whichever CTA arrives last
        const int x = i < gamma ? __ldg(p.tokens + (size_t)s * gamma + i) : -1;
        const int badtok = (i < gamma) && (x < 0 || x >= V);
        const bool has_x = !GREEDY && i < gamma && !badtok;
        float zt = 0.f, zd = 0.f, r = 0.f;
        if (lane == 1 && has_x) zt = load_logit<DT>(trow, x);
        if (lane == 2 && has_x) zd = load_logit<DT>(drow, x);
        if (lane == 3 && has_x) r = __ldg(p.uniforms + (size_t)s * (gamma + 1) + i);
        const int prev_bad = (i == 0) ? 0 : __ldcg(&w.st[s].bad);
        if constexpr (GREEDY) {
          AM a = am_empty();
          for (int q = lane; q < NC; q += 32) {
            const MS *qq = w.part + ((size_t)s * NC + q) * 2;
            AM b;
            b.v = __ldcg(reinterpret_cast<const float *>(qq));
            b.i = __ldcg(reinterpret_cast<const int *>(qq) + 1);
            b.bad = __ldcg(reinterpret_cast<const int *>(qq) + 2);
            a = am_merge(a, b);
          }
          a = warp_down_am(a);
          if (lane == 0) {
            w.cnt[s] = 0;
            const int bad = prev_bad | badtok;
            const bool invalid = a.bad || !(a.v > -kInf);
            const bool acc = !invalid && i < gamma && x == a.i;
            if (p.out_accept && i < gamma && !invalid)
              p.out_accept[(size_t)s * gamma + i] = acc ? 1.f : 0.f;
            if (invalid) {
              finish(s, -1, -1, 0.f, SD_DEV_NONFINITE | (bad ? SD_DEV_BAD_TOKEN : 0), i);
            } else if (acc) {
              w.st[s].bad = bad;
              w.act[((i + 1) & 1) * p.B + atomicAdd(&w.act_n[i + 1], 1)] = s;
            } else {
              finish(s, i, a.i, 1.f, bad ? SD_DEV_BAD_TOKEN : 0, i + 1);
            }
          }
        } else {
          MS mt = ms_empty(), md = ms_empty();
          for (int q = lane; q < NC; q += 32) {
            const MS *qq = w.part + ((size_t)s * NC + q) * 2;
            MS a{__ldcg(&qq[0].m), __ldcg(&qq[0].s)};
            MS b{__ldcg(&qq[1].m), __ldcg(&qq[1].s)};
            mt = ms_merge(mt, a, k2);
            md = ms_merge(md, b, k2);
          }
          mt = warp_down_ms(mt, k2);
          md = warp_down_ms(md, k2);
          zt = __shfl_sync(0xffffffffu, zt, 1);
          zd = __shfl_sync(0xffffffffu, zd, 2);
          r = __shfl_sync(0xffffffffu, r, 3);
          if (lane == 0) {
            w.cnt[s] = 0;
            const int bad = prev_bad | badtok;
            const bool invalid = !ms_valid(mt) || (has_d && !ms_valid(md));
            bool acc = false;
            float accp = 0.f;
            if (!invalid && has_x) {
              const float e = fmaf(zt, k2, -mt.m * k2) - fmaf(zd, k2, -md.m * k2);
              const float rho = exp2f(e) * (md.s / mt.s);
              acc = r <= rho;
              accp = fminf(1.f, rho);
            }
            if (p.out_accept && i < gamma && !invalid)
              p.out_accept[(size_t)s * gamma + i] = accp;
            if (invalid) {
              finish(s, -1, -1, 0.f, SD_DEV_NONFINITE | (bad ? SD_DEV_BAD_TOKEN : 0), i);
            } else if (acc) {
              w.st[s].bad = bad;
              w.act[((i + 1) & 1) * p.B + atomicAdd(&w.act_n[i + 1], 1)] = s;
            } else {  // rejection at i, or the bonus at i == gamma
              SeqState q;
              q.mt = mt;
              q.md = md;
              q.n = i;
              q.bad = bad;
              w.st[s] = q;
              w.drw[((i + 1) & 1) * p.B + atomicAdd(&w.drw_n[i + 1], 1)] = s;
            }
          }
        }
      }
      __syncthreads();
    } else {
      // ---------------- draw item: chunk mass of the weights -------------
      const int e = w.drw[(i & 1) * p.B + (idx - A)];
      const int s = e & 0x3fffffff;
      const bool ponly = (e >> 30) & 1;
      const SeqState q = w.st[s];
      const int n = q.n;
      const bool has_q = (n < gamma) && !ponly;
      const char *trow = tbase + ((size_t)s * (gamma + 1) + n) * rowb;
      const char *drow =
          has_q ? dbase + ((size_t)s * p.d_seq_rows + n) * rowb : trow;
      Weight W;
      W.k2 = k2;
      W.mtk = q.mt.m * k2;
      W.ist = 1.f / q.mt.s;
      W.mdk = q.md.m * k2;
      W.cq = 1.f / q.md.s;
      ring_mass<DT, VW>(rg, trow, drow, has_q, W, cs, segmass);
      __syncthreads();
      slice_prefix(segmass, cs.nseg, sh.draw.chunk_pre);
      __syncthreads();
      if (tid == 0) w.dmass[(size_t)s * NC + c] = cs.nseg ? sh.draw.chunk_pre[31] : 0.0;
      if (!last_arrival(&w.dcnt[s], NC)) continue;
      // ---- this CTA completes the draw: total, crossing chunk, scan -------
      if (warp == 0) {
        // lane l holds chunks l, l+32, ...; running sums in chunk order
        const float u = __ldg(p.uniforms + (size_t)s * (gamma + 1) + gamma);
        double run = 0.0, tau = 0.0, bef = 0.0, lastbef = 0.0;
        int own = -1, lastpos = -1;
        for (int base = 0; base < NC; base += 32) {
          const int k = base + lane;
          const double m = k < NC ? __ldcg(&w.dmass[(size_t)s * NC + k]) : 0.0;
          for (int l = 0; l < 32 && base + l < NC; ++l) {
            const double ml = __shfl_sync(0xffffffffu, m, l);
            run += ml;  // every lane keeps the same running sum
          }
        }
        const double tot = run;
        tau = (double)u * tot;
        run = 0.0;
        for (int base = 0; base < NC; base += 32) {
          const int k = base + lane;
          const double m = k < NC ? __ldcg(&w.dmass[(size_t)s * NC + k]) : 0.0;
          for (int l = 0; l < 32 && base + l < NC; ++l) {
            const double ml = __shfl_sync(0xffffffffu, m, l);
            if (own < 0 && run + ml > tau) {
              own = base + l;
              bef = run;
            }
            if (ml > 0.0) {
              lastpos = base + l;
              lastbef = run;
            }
            run += ml;
          }
        }
        if (own < 0 && tot > 0.0) {  // rounding: last chunk with mass
          own = lastpos;
          bef = lastbef;
        }
        if (lane == 0) {
          w.dcnt[s] = 0;
          sh.draw.N = tot;
          sh.draw.owner = tot > 0.0 ? own : -1;
          sh.draw.tau = tau - bef;
        }
      }
      __syncthreads();
      if (sh.draw.owner < 0) {
        // zero residual mass: queue a draw from p_n for the next level
        if (tid == 0)
          w.drw[((i + 1) & 1) * p.B + atomicAdd(&w.drw_n[i + 1], 1)] =
              s | (1 << 30);
        continue;
      }
      const Slice ps = chunk_slice(sh.draw.owner);
      const double N = sh.draw.N;
      ring_mass<DT, VW>(rg, trow, drow, has_q, W, ps, segmass);
      __syncthreads();
      slice_prefix(segmass, ps.nseg, sh.draw.chunk_pre);
      __syncthreads();
      if (tid == 0) {
        double tin = 0.0;
        sh.draw.seg = find_segment(segmass, ps.nseg, sh.draw.chunk_pre,
                                   sh.draw.tau, &tin);
        sh.draw.tau_seg = (float)tin;
      }
      __syncthreads();
      if (warp == 0) {
        const GRow<DT, VW> ra{trow}, rb{drow};
        const int sg = sh.draw.seg;
        const int v = ps.vbeg + sg * 32 + lane;
        float wv[VW];
        if (v < ps.vend) {
          weights<DT, VW>(ra.get(v), rb.get(v), has_q, W, wv);
        } else {
#pragma unroll
          for (int k = 0; k < VW; ++k) wv[k] = 0.f;
        }
        float wt;
        const int t = warp_pick<VW>(wv, sh.draw.tau_seg, (ps.vbeg + sg * 32) * VW, &wt);
        if (lane == 0)
          finish(s, n, t, (float)((double)wt / N),
                 (q.bad ? SD_DEV_BAD_TOKEN : 0) | (ponly ? SD_DEV_ZERO_MASS : 0),
                 n + 1);
      }
      __syncthreads();
    }
  }
}

using WideKernel = void (*)(const WideParams);

static WideKernel pick_wide(int dt, bool greedy) {
  if (dt == SD_F32) return greedy ? wide_level_kernel<0, 4, true> : wide_level_kernel<0, 4, false>;
  return greedy ? wide_level_kernel<1, 8, true> : wide_level_kernel<1, 8, false>;
}

// chunk of ~8192 elements per row (32 KB fp32 / 16 KB bf16)
static int wide_chunk_vecs(int dt) { return dt == SD_F32 ? 2048 : 1024; }

static size_t align256(size_t x) { return (x + 255) / 256 * 256; }

size_t wide_workspace(int B, int gamma, int V, sd_dtype dt) {
  const int vw = dt == SD_F32 ? 4 : 8;
  const int nvec = V / vw;
  const int cv = wide_chunk_vecs(dt);
  const int NC = (nvec + cv - 1) / cv;
  const int L = gamma + 4;
  size_t b = 0;
  b += align256(sizeof(int) * L * 2);          // act_n, drw_n
  b += align256(sizeof(int) * 2 * B) * 2;      // act, drw
  b += align256(sizeof(int) * B) * 2;          // cnt, dcnt
  b += align256(sizeof(MS) * (size_t)B * NC * 2);
  b += align256(sizeof(double) * (size_t)B * NC);
  b += align256(sizeof(SeqState) * B);
  return b;
}

// The counters (act_n, drw_n, cnt, dcnt) start at zero: one memset of the
// leading part of the workspace per call.
sd_status wide_launch(const void *target, const void *draft, sd_dtype dt,
                      long long d_seq_rows, const int32_t *tokens, const float *uniforms, int B,
                      int gamma, int V, float T, int32_t *n_acc,
                      int32_t *out_tokens, float *out_prob, float *out_accept,
                      int32_t *dev_status, void *ws, size_t ws_bytes,
                      cudaStream_t stream) {
  int sms = 0;
  sd_status st = check_device(&sms);
  if (st != SD_OK) return st;
  const size_t need = wide_workspace(B, gamma, V, dt);
  if (!ws || ws_bytes < need)
    return fail(SD_ERR_INVALID_ARG, "workspace of >= %zu bytes required",
                need);
  const bool greedy = (T == 0.f);
  const int vw = dt == SD_F32 ? 4 : 8;
  const int nvec = V / vw;
  const int cv = wide_chunk_vecs(dt);
  const int NC = (nvec + cv - 1) / cv;
  const int L = gamma + 4;
  char *b = static_cast<char *>(ws);
  WideWs w;
  w.act_n = reinterpret_cast<int *>(b);
  w.drw_n = w.act_n + L;
  b += align256(sizeof(int) * L * 2);
  int *cnt = reinterpret_cast<int *>(b);
  w.cnt = cnt;
  b += align256(sizeof(int) * B);
  w.dcnt = reinterpret_cast<int *>(b);
  b += align256(sizeof(int) * B);
  const size_t zero_bytes = (size_t)(b - static_cast<char *>(ws));
  w.act = reinterpret_cast<int *>(b);
  b += align256(sizeof(int) * 2 * B);
  w.drw = reinterpret_cast<int *>(b);
  b += align256(sizeof(int) * 2 * B);
  w.part = reinterpret_cast<MS *>(b);
  b += align256(sizeof(MS) * (size_t)B * NC * 2);
  w.dmass = reinterpret_cast<double *>(b);
  b += align256(sizeof(double) * (size_t)B * NC);
  w.st = reinterpret_cast<SeqState *>(b);
  SDV_CUDA(cudaMemsetAsync(ws, 0, zero_bytes, stream));

  WideKernel kern = pick_wide(dt, greedy);
  const size_t seg_bytes = ((size_t)((cv + 31) / 32) * 4 + 127) / 128 * 128;
  const size_t smem = seg_bytes + kRingBytes;
  int maxc = 0;
  st = max_active_clusters((const void *)kern, 1, smem, &maxc);
  if (st != SD_OK) return st;
  WideParams prm;
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
  prm.dev_status = dev_status;
  prm.NC = NC;
  prm.chunk_vecs = cv;
  prm.seg_bytes = (int)seg_bytes;
  prm.ws = w;
  const int levels = greedy ? gamma + 1 : gamma + 3;
  for (int lv = 0; lv < levels; ++lv) {
    prm.level = lv;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)maxc, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = lv > 0 ? 1 : 0;
    void *args[] = {&prm};
    SDV_CUDA(cudaLaunchKernelExC(&cfg, (const void *)kern, args));
  }
  return SD_OK;
}

}  // namespace sdv
