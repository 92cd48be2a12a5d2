/*
 * sd_oracle.c -- plain, slow, fp64 CPU oracle for the verify step of
 * speculative decoding.  TEST INFRASTRUCTURE ONLY: it is called by the test
 * suite, by the smoke check and by the CPU-baseline leg of the benchmark,
 * never by the product path.  It shares no source with the CUDA library.
 *
 * Every function follows the pages step by step, in double precision, with
 * no blocking, fusion or reordering:
 *
 *  - "01 · Draft-then-verify" (llm-infra-atlas), section 1, Algorithm 1:
 *    draft gamma tokens, one target pass gives p_1..p_{gamma+1}, scan left
 *    to right drawing r_i and rejecting at the first r_i > p_i(x_i)/q_i(x_i),
 *    then sample a correction from norm(max(0, p_{n+1} - q_{n+1})) or, when
 *    every draft is accepted, a bonus token from p_{gamma+1}.
 *  - same page, section 2.1: single-step accept probability min(1, p/q) and
 *    the residual p' = norm(max(0, p - q)).
 *  - same page, section 2.2: greedy (temperature 0) reduces to comparing the
 *    draft id with argmax p.
 *  - same page, section 4, the spec_step listing: 0-based indexing, ps[n]
 *    minus qs[n] for the residual, ps[gamma] for the bonus.
 *  - SpecDiff-2 (MLSys'26), "core method", self-selection acceptance: K
 *    candidate drafts from shared position-wise marginals, the verifier keeps
 *    the candidate with the longest accepted streak.
 *  - PRESTO, section 2.1 "tree-based speculative decoding": prefix-wise
 *    verification from the root, acceptance factorised along the path.
 *  - PRESTO, section 4.1 (prefix-aligned score s = log q_d + lambda log
 *    rho_d, path score S(P), Eq. 10), section 4.2 and Algorithm 1 (beam
 *    search with global retention under a node budget), section 4.4 (the
 *    score is the log of the KL-regularised proxy q rho^lambda / Z).
 *  - SpecBranch, branch resampling: k = max(1, floor(k_max (1 - q(x_b))))
 *    branches, the Top-k of the draft distribution at the branch point.
 *  - SpecDiff-2, "core method", greedy acceptance: a drafted token is
 *    accepted with the verifier's probability of it, independently of the
 *    drafter, and a rejected position is resampled from the residual.
 *  - Speculative Speculative Decoding / Saguaro, "speculation cache
 *    strategy": Definition 11 (power-law cache miss) and Theorem 12
 *    (geometric fan-out F_k = F_0 a^{k/(1+r)}, capped at position K), and
 *    the top-F_k-per-position cache fill; "technical architecture": the
 *    speculator serves the next round from its cache when the verification
 *    outcome (k accepted, then t*) is in the cache.
 *
 * Readings where the pages are silent (all listed in the design notes):
 *  - accept iff r <= p(x)/q(x) (reject on '>', Algorithm 1 step 3);
 *  - p = softmax(z / T) for target and draft with the same T; T == 0 is
 *    greedy on the raw logits (lowest index wins a tie);
 *  - inverse CDF: the smallest j with C_j > u * N (strict), C_j the running
 *    sum of the weights in index order; if rounding leaves no such j, the
 *    last j with positive weight;
 *  - a residual of exactly zero mass falls back to sampling p and sets
 *    status bit 8;
 *  - filtered sampling ("01 · Draft-then-verify", section 4, standardised
 *    sampling: top-k / nucleus act on p and q before the ratio): softmax at
 *    temperature T, keep the top_k tokens by (logit desc, index asc), then
 *    the smallest prefix of them, in that order, whose renormalised mass
 *    reaches top_p, and renormalise over what is kept;
 *  - a draft token outside [0, V) is a rejection (status bit 1);
 *  - a row holding NaN or +inf, or only -inf, makes its sequence invalid
 *    (status bit 2; n = -1, every token -1);
 *  - a parent array with parent[0] != -1 or parent[v] outside [0, v) makes
 *    its tree invalid (status bit 4);
 *  - tree siblings are tried in increasing node index against the fixed
 *    draft row of their parent, with p <- norm(max(0, p - q)) after each
 *    rejection; the final draw of a tree uses uniform slot 0;
 *  - greedy acceptance is read as Algorithm 1 with the draft distribution
 *    the point mass on the drafted token (the deterministic-draft tree
 *    rule): accept iff r <= p(x), residual = p with x removed and
 *    renormalised, siblings tried in increasing node index;
 *  - K candidates as one tree: candidate k's token at position j is node
 *    1 + j K + k, below the node of its prefix; a token repeated under the
 *    same prefix is a leaf duplicate (the sibling rule must see every iid
 *    draw) and the candidate continues below the first copy; a node takes
 *    the target row of the candidate that created it;
 *  - PRESTO construction, one depth per call: each frontier path proposes
 *    its b tokens of largest s (ties to the lower id, s = -inf excluded);
 *    all proposals are ordered by (S + s desc, path slot asc, token asc)
 *    and added while the budget lasts; the first W added form the next
 *    frontier; rho is given (log rho rows), its learned predictor is not
 *    part of this;
 *  - SpecBranch fork: q(x_b) is the drafted token's probability under
 *    softmax(z / T) (the point mass on the argmax at T == 0); k is capped
 *    at V; the branches are ordered by (logit desc, id asc);
 *  - kcand selection: the largest accepted count, ties to the lowest k; the
 *    final draw uses uniform slot [b][k*][gamma];
 *  - fan-out integerisation: floor of F_0 w_k, the remainder handed out by
 *    largest fractional part, ties to the lower k; top-F orders by
 *    (value descending, index ascending), -0 equal to +0.
 *
 * Every draw also records a margin: |r - p/q| for an accept test (the
 * smallest over the tests of a sequence) and the distance of u to the two
 * CDF boundaries of the chosen token for the inverse-CDF draw, plus the
 * range of tokens whose CDF interval lies within ORC_BAND of u.  The margins
 * tell the tests where a finite-precision implementation may legitimately
 * disagree, and the range which tokens it may then return.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_BF16 1

#define ORC_ST_BAD_TOKEN 1
#define ORC_ST_NONFINITE 2
#define ORC_ST_BAD_PARENT 4
#define ORC_ST_ZERO_MASS 8

/* ---- input access: fp32 as is, bf16 widened exactly (it is the top half
 * of an fp32 bit pattern) ---- */
static double logit_at(const void *base, int dtype, size_t i) {
  if (dtype == ORC_F32) return (double)((const float *)base)[i];
  uint32_t w = (uint32_t)((const uint16_t *)base)[i] << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* A row is usable iff no entry is NaN or +inf and at least one entry is
 * finite.  Returns 1 if usable. */
static int row_ok(const void *base, int dtype, size_t off, int V) {
  int any_finite = 0;
  for (int j = 0; j < V; ++j) {
    double z = logit_at(base, dtype, off + (size_t)j);
    if (isnan(z) || z == INFINITY) return 0;
    if (z > -INFINITY) any_finite = 1;
  }
  return any_finite;
}

/* p = softmax(z / T), T > 0, with max subtraction.  Returns 0 on an
 * unusable row. */
static int softmax_row(const void *base, int dtype, size_t off, int V,
                       double T, double *p) {
  if (!row_ok(base, dtype, off, V)) return 0;
  double m = -INFINITY;
  for (int j = 0; j < V; ++j) {
    double z = logit_at(base, dtype, off + (size_t)j);
    if (z > m) m = z;
  }
  double Z = 0.0;
  for (int j = 0; j < V; ++j) {
    p[j] = exp((logit_at(base, dtype, off + (size_t)j) - m) / T);
    Z += p[j];
  }
  for (int j = 0; j < V; ++j) p[j] /= Z;
  return 1;
}

/* argmax over the raw logits, lowest index on ties.  -1 on an unusable row. */
static int argmax_row(const void *base, int dtype, size_t off, int V) {
  if (!row_ok(base, dtype, off, V)) return -1;
  int best = 0;
  double bv = logit_at(base, dtype, off);
  for (int j = 1; j < V; ++j) {
    double z = logit_at(base, dtype, off + (size_t)j);
    if (z > bv) { bv = z; best = j; }
  }
  return best;
}

/* Inverse-CDF draw from the weights w (not necessarily normalised, total
 * N > 0): the smallest j with C_j > u N.  Writes w_t / N, the margin
 * min(|u - C_{t-1}/N|, |u - C_t/N|), and the range [lo, hi] of every token
 * whose interval [C_{j-1}/N, C_j/N] comes within ORC_BAND of u: the tokens a
 * correct finite-precision draw may return. */
#define ORC_BAND 1e-5
#define SD_ORC_MAX_GAMMA 64 /* longest draft the filtered verify takes */
static int sample_icdf(const double *w, int V, double u, double *prob,
                       double *margin, int *lo, int *hi) {
  double N = 0.0;
  for (int j = 0; j < V; ++j) N += w[j];
  double target = u * N;
  double C = 0.0, Cprev = 0.0;
  int t = -1;
  for (int j = 0; j < V; ++j) {
    Cprev = C;
    C += w[j];
    if (C > target) { t = j; break; }
  }
  if (t < 0) { /* rounding left no crossing: last token with mass */
    for (int j = V - 1; j >= 0; --j)
      if (w[j] > 0.0) { t = j; break; }
    C = N;
    Cprev = N - w[t];
  }
  *prob = w[t] / N;
  double m1 = fabs(u - Cprev / N), m2 = fabs(u - C / N);
  *margin = m1 < m2 ? m1 : m2;
  /* walk outwards while neighbouring intervals touch [u - band, u + band] */
  int a = t;
  double left = Cprev; /* C_{a-1} */
  while (a > 0 && left / N > u - ORC_BAND) {
    --a;
    left -= w[a];
  }
  int b = t;
  double right = C; /* C_b */
  while (b < V - 1 && right / N < u + ORC_BAND) {
    ++b;
    right += w[b];
  }
  *lo = a;
  *hi = b;
  return t;
}

/* The accept ratio p(x)/q(x); 0 when p(x) == 0, +inf when only q(x) == 0. */
static double accept_ratio(double px, double qx) {
  if (px == 0.0) return 0.0;
  if (qx == 0.0) return INFINITY;
  return px / qx;
}

static void note_margin(double *margin, double m) {
  if (m < *margin) *margin = m;
}

/* One accept test r <= rho: counted in *tests; its margin |r - rho| noted
 * (there is none when rho is infinite: q(x) == 0 < p(x) always accepts),
 * and counted in *flagged when that margin is below ORC_BAND. */
static void note_test(double *margin, int *tests, int *flagged, double r,
                      double rho) {
  ++*tests;
  if (!isfinite(rho)) return;
  const double m = fabs(r - rho);
  note_margin(margin, m);
  if (m < ORC_BAND) ++*flagged;
}

/* Per-sequence test counts (nullable outputs): none for greedy or invalid
 * sequences, whose margins are infinite too. */
static void put_tests(int32_t *acc_tests, int32_t *acc_flagged, int b,
                      int none, int nt, int nf) {
  if (acc_tests) acc_tests[b] = none ? 0 : nt;
  if (acc_flagged) acc_flagged[b] = none ? 0 : nf;
}

/* ------------------------------------------------------------------------
 * Linear verify ("01 · Draft-then-verify", Algorithm 1 and spec_step).
 * target [B, gamma+1, V], draft [B, gamma, V] (unused when T == 0),
 * tokens [B, gamma], uniforms [B, gamma+1] (slot gamma is the final draw).
 * out_accept [B, gamma]: min(1, p/q) of each evaluated test (1/0 when
 * T == 0), -1 where no test was made.  out_resid [B, V] (nullable): the
 * normalised distribution the last token was drawn from.
 * ---------------------------------------------------------------------- */
int orc_verify_linear(const void *target, const void *draft, int dtype,
                      const int32_t *tokens, const float *uniforms, int B,
                      int gamma, int V, double T, int32_t *n_acc,
                      int32_t *out_tokens, double *out_prob,
                      double *out_accept, double *margin_acc,
                      double *margin_cdf, int32_t *cdf_lo, int32_t *cdf_hi,
                      int32_t *acc_tests, int32_t *acc_flagged,
                      double *out_resid, int32_t *status) {
  double *p = malloc(sizeof(double) * (size_t)V);
  double *q = malloc(sizeof(double) * (size_t)V);
  double *w = malloc(sizeof(double) * (size_t)V);
  if (!p || !q || !w) { free(p); free(q); free(w); return 1; }
  const int G1 = gamma + 1;
  for (int b = 0; b < B; ++b) {
    int st = 0, n = 0, t = -1, invalid = 0, lo = -1, hi = -1, nt = 0, nf = 0;
    double mg = INFINITY, mc = INFINITY, prob = 0.0;
    for (int i = 0; i < gamma; ++i) out_accept[(size_t)b * gamma + i] = -1.0;
    if (T == 0.0) {
      for (int i = 0; i < gamma; ++i) {
        int a = argmax_row(target, dtype, ((size_t)b * G1 + i) * V, V);
        if (a < 0) { invalid = 1; break; }
        int x = tokens[(size_t)b * gamma + i];
        if (x < 0 || x >= V) st |= ORC_ST_BAD_TOKEN;
        int ok = (x == a);
        out_accept[(size_t)b * gamma + i] = ok ? 1.0 : 0.0;
        if (!ok) break;
        ++n;
      }
      if (!invalid) {
        t = argmax_row(target, dtype, ((size_t)b * G1 + n) * V, V);
        if (t < 0) invalid = 1;
        prob = 1.0;
        lo = hi = t;
        if (out_resid && !invalid) {
          for (int j = 0; j < V; ++j) out_resid[(size_t)b * V + j] = 0.0;
          out_resid[(size_t)b * V + t] = 1.0;
        }
      }
    } else {
      int rejected = 0;
      for (int i = 0; i < gamma; ++i) {
        if (!softmax_row(target, dtype, ((size_t)b * G1 + i) * V, V, T, p) ||
            !softmax_row(draft, dtype, ((size_t)b * gamma + i) * V, V, T, q)) {
          invalid = 1;
          break;
        }
        int x = tokens[(size_t)b * gamma + i];
        double r = (double)uniforms[(size_t)b * G1 + i];
        int ok;
        if (x < 0 || x >= V) {
          st |= ORC_ST_BAD_TOKEN;
          ok = 0;
          out_accept[(size_t)b * gamma + i] = 0.0;
        } else {
          double rho = accept_ratio(p[x], q[x]);
          note_test(&mg, &nt, &nf, r, rho);
          ok = (r <= rho);
          out_accept[(size_t)b * gamma + i] = rho < 1.0 ? rho : 1.0;
        }
        if (!ok) { rejected = 1; break; }
        ++n;
      }
      if (!invalid) {
        if (rejected) { /* residual norm(max(0, p_n - q_n)) */
          double N = 0.0;
          for (int j = 0; j < V; ++j) {
            double d = p[j] - q[j];
            w[j] = d > 0.0 ? d : 0.0;
            N += w[j];
          }
          if (N == 0.0) { /* nothing left to correct with: sample p_n */
            st |= ORC_ST_ZERO_MASS;
            for (int j = 0; j < V; ++j) w[j] = p[j];
          }
        } else { /* bonus from p_{gamma+1} */
          if (!softmax_row(target, dtype, ((size_t)b * G1 + gamma) * V, V, T,
                           p))
            invalid = 1;
          else
            for (int j = 0; j < V; ++j) w[j] = p[j];
        }
      }
      if (!invalid) {
        double u = (double)uniforms[(size_t)b * G1 + gamma];
        t = sample_icdf(w, V, u, &prob, &mc, &lo, &hi);
        if (out_resid) {
          double N = 0.0;
          for (int j = 0; j < V; ++j) N += w[j];
          for (int j = 0; j < V; ++j) out_resid[(size_t)b * V + j] = w[j] / N;
        }
      }
    }
    if (invalid) {
      st |= ORC_ST_NONFINITE;
      n = -1;
      prob = 0.0;
      mg = mc = INFINITY;
      lo = hi = -1;
    }
    n_acc[b] = n;
    for (int i = 0; i < G1; ++i) {
      int32_t v = -1;
      if (!invalid) {
        if (i < n) v = tokens[(size_t)b * gamma + i];
        else if (i == n) v = t;
      }
      out_tokens[(size_t)b * G1 + i] = v;
    }
    out_prob[b] = prob;
    margin_acc[b] = (T == 0.0) ? INFINITY : mg;
    margin_cdf[b] = (T == 0.0) ? INFINITY : mc;
    cdf_lo[b] = lo;
    cdf_hi[b] = hi;
    put_tests(acc_tests, acc_flagged, b, T == 0.0 || invalid, nt, nf);
    status[b] = st;
  }
  free(p); free(q); free(w);
  return 0;
}

/* ------------------------------------------------------------------------
 * K-candidate verify with verifier self-selection (SpecDiff-2, "core
 * method").  target [B, K, gamma+1, V]: candidate k's own target rows;
 * draft [B, gamma, V]: the position-wise marginals shared by all K
 * candidates; tokens [B, K, gamma]; uniforms [B, K, gamma+1].
 * Each candidate is scanned with the linear rule; the selected candidate is
 * the one with the most accepted tokens (lowest k on ties); its residual
 * or bonus draw uses uniform [b][k*][gamma].
 * ---------------------------------------------------------------------- */
int orc_verify_kcand(const void *target, const void *draft, int dtype,
                     const int32_t *tokens, const float *uniforms, int B,
                     int K, int gamma, int V, double T, int32_t *n_acc,
                     int32_t *sel_k, int32_t *out_tokens, int32_t *n_per_cand,
                     double *out_prob, double *margin_acc,
                     double *margin_cdf, int32_t *cdf_lo, int32_t *cdf_hi,
                     int32_t *acc_tests, int32_t *acc_flagged,
                     int32_t *status) {
  double *p = malloc(sizeof(double) * (size_t)V);
  double *q = malloc(sizeof(double) * (size_t)V);
  double *w = malloc(sizeof(double) * (size_t)V);
  if (!p || !q || !w) { free(p); free(q); free(w); return 1; }
  const int G1 = gamma + 1;
#define TROW(b, k, j) ((((size_t)(b) * K + (k)) * G1 + (j)) * (size_t)V)
#define DROW(b, j) (((size_t)(b) * gamma + (j)) * (size_t)V)
  for (int b = 0; b < B; ++b) {
    int st = 0, invalid = 0, lo = -1, hi = -1, nt = 0, nf = 0;
    double mg = INFINITY, mc = INFINITY, prob = 0.0;
    int best_k = 0, best_n = -1, t = -1;
    for (int k = 0; k < K && !invalid; ++k) {
      int n = 0;
      for (int j = 0; j < gamma; ++j) {
        int x = tokens[((size_t)b * K + k) * gamma + j];
        int ok;
        if (T == 0.0) {
          int a = argmax_row(target, dtype, TROW(b, k, j), V);
          if (a < 0) { invalid = 1; break; }
          if (x < 0 || x >= V) st |= ORC_ST_BAD_TOKEN;
          ok = (x == a);
        } else {
          if (!softmax_row(target, dtype, TROW(b, k, j), V, T, p) ||
              !softmax_row(draft, dtype, DROW(b, j), V, T, q)) {
            invalid = 1;
            break;
          }
          if (x < 0 || x >= V) {
            st |= ORC_ST_BAD_TOKEN;
            ok = 0;
          } else {
            double r = (double)uniforms[((size_t)b * K + k) * G1 + j];
            double rho = accept_ratio(p[x], q[x]);
            note_test(&mg, &nt, &nf, r, rho);
            ok = (r <= rho);
          }
        }
        if (!ok) break;
        ++n;
      }
      if (invalid) break;
      n_per_cand[(size_t)b * K + k] = n;
      if (n > best_n) { best_n = n; best_k = k; }
    }
    if (!invalid) {
      const int n = best_n, k = best_k;
      if (T == 0.0) {
        t = argmax_row(target, dtype, TROW(b, k, n), V);
        if (t < 0) invalid = 1;
        prob = 1.0;
        lo = hi = t;
      } else {
        if (n < gamma) {
          if (!softmax_row(target, dtype, TROW(b, k, n), V, T, p) ||
              !softmax_row(draft, dtype, DROW(b, n), V, T, q))
            invalid = 1;
          else {
            double N = 0.0;
            for (int j = 0; j < V; ++j) {
              double d = p[j] - q[j];
              w[j] = d > 0.0 ? d : 0.0;
              N += w[j];
            }
            if (N == 0.0) {
              st |= ORC_ST_ZERO_MASS;
              for (int j = 0; j < V; ++j) w[j] = p[j];
            }
          }
        } else {
          if (!softmax_row(target, dtype, TROW(b, k, gamma), V, T, p))
            invalid = 1;
          else
            for (int j = 0; j < V; ++j) w[j] = p[j];
        }
        if (!invalid) {
          double u = (double)uniforms[((size_t)b * K + k) * G1 + gamma];
          t = sample_icdf(w, V, u, &prob, &mc, &lo, &hi);
        }
      }
    }
    if (invalid) {
      st |= ORC_ST_NONFINITE;
      for (int k = 0; k < K; ++k) n_per_cand[(size_t)b * K + k] = -1;
      n_acc[b] = -1;
      sel_k[b] = -1;
      prob = 0.0;
      mg = mc = INFINITY;
      lo = hi = -1;
    } else {
      n_acc[b] = best_n;
      sel_k[b] = best_k;
    }
    for (int i = 0; i < G1; ++i) {
      int32_t v = -1;
      if (!invalid) {
        if (i < best_n) v = tokens[((size_t)b * K + best_k) * gamma + i];
        else if (i == best_n) v = t;
      }
      out_tokens[(size_t)b * G1 + i] = v;
    }
    out_prob[b] = prob;
    margin_acc[b] = (T == 0.0) ? INFINITY : mg;
    margin_cdf[b] = (T == 0.0) ? INFINITY : mc;
    cdf_lo[b] = lo;
    cdf_hi[b] = hi;
    put_tests(acc_tests, acc_flagged, b, T == 0.0 || invalid, nt, nf);
    status[b] = st;
  }
#undef TROW
#undef DROW
  free(p); free(q); free(w);
  return 0;
}

/* ------------------------------------------------------------------------
 * Tree verify.  target [B, N, V]: row u is p(. | path to u); draft [B, N, V]:
 * row u is the q that drafted u's children.  parent [B, N] with parent[0]
 * == -1 and parent[v] < v; node_tokens [B, N] (slot 0 unused); uniforms
 * [B, N]: slot v tests node v, slot 0 is the final draw.
 * The walk starts at the root; the children of the current node are tried
 * in increasing node index; each rejection replaces p by norm(max(0, p-q))
 * with q the parent's draft row; an accepted child becomes the current node
 * with fresh rows.  When no child is accepted (or at a leaf) the last token
 * is drawn from the current p.
 * Outputs: n_acc = number of accepted nodes; out_nodes [B, N] the accepted
 * path (-1 padded); out_tokens [B, N] the accepted tokens then the final
 * token (-1 padded).
 * ---------------------------------------------------------------------- */
int orc_verify_tree(const void *target, const void *draft, int dtype,
                    const int32_t *parent, const int32_t *node_tokens,
                    const float *uniforms, int B, int N, int V, double T,
                    int32_t *n_acc, int32_t *out_tokens, int32_t *out_nodes,
                    double *out_prob, double *margin_acc, double *margin_cdf,
                    int32_t *cdf_lo, int32_t *cdf_hi, int32_t *acc_tests,
                    int32_t *acc_flagged, int32_t *status) {
  double *p = malloc(sizeof(double) * (size_t)V);
  double *q = malloc(sizeof(double) * (size_t)V);
  if (!p || !q) { free(p); free(q); return 1; }
  for (int b = 0; b < B; ++b) {
    const int32_t *par = parent + (size_t)b * N;
    const int32_t *tok = node_tokens + (size_t)b * N;
    const float *U = uniforms + (size_t)b * N;
    int st = 0, invalid = 0, depth = 0, t = -1, lo = -1, hi = -1;
    int nt = 0, nf = 0;
    double mg = INFINITY, mc = INFINITY, prob = 0.0;
    for (int i = 0; i < N; ++i) {
      out_nodes[(size_t)b * N + i] = -1;
      out_tokens[(size_t)b * N + i] = -1;
    }
    if (par[0] != -1) invalid = 4;
    for (int v = 1; v < N && !invalid; ++v)
      if (par[v] < 0 || par[v] >= v) invalid = 4;
    int cur = 0;
    while (!invalid) {
      size_t off = ((size_t)b * N + cur) * (size_t)V;
      int has_child = 0;
      for (int v = cur + 1; v < N; ++v)
        if (par[v] == cur) { has_child = 1; break; }
      int next = -1;
      if (T == 0.0) {
        int a = argmax_row(target, dtype, off, V);
        if (a < 0) { invalid = 2; break; }
        for (int v = cur + 1; v < N; ++v) {
          if (par[v] != cur) continue;
          if (tok[v] < 0 || tok[v] >= V) st |= ORC_ST_BAD_TOKEN;
          if (tok[v] == a) { next = v; break; }
        }
        if (next < 0) { t = a; prob = 1.0; lo = hi = a; break; }
      } else {
        if (!softmax_row(target, dtype, off, V, T, p)) { invalid = 2; break; }
        if (has_child && !softmax_row(draft, dtype, off, V, T, q)) {
          invalid = 2;
          break;
        }
        int zero_mass = 0;
        for (int v = cur + 1; v < N && next < 0 && !zero_mass; ++v) {
          if (par[v] != cur) continue;
          int x = tok[v];
          int ok = 0;
          if (x < 0 || x >= V) {
            st |= ORC_ST_BAD_TOKEN;
          } else {
            double rho = accept_ratio(p[x], q[x]);
            note_test(&mg, &nt, &nf, (double)U[v], rho);
            ok = ((double)U[v] <= rho);
          }
          if (ok) { next = v; break; }
          /* rejected: p <- norm(max(0, p - q)) */
          double S = 0.0;
          for (int j = 0; j < V; ++j) {
            double d = p[j] - q[j];
            p[j] = d > 0.0 ? d : 0.0;
            S += p[j];
          }
          if (S == 0.0) { /* fall back to the un-subtracted p of this node */
            st |= ORC_ST_ZERO_MASS;
            softmax_row(target, dtype, off, V, T, p);
            zero_mass = 1;
          } else {
            for (int j = 0; j < V; ++j) p[j] /= S;
          }
        }
        if (next < 0) {
          t = sample_icdf(p, V, (double)U[0], &prob, &mc, &lo, &hi);
          break;
        }
      }
      out_nodes[(size_t)b * N + depth] = next;
      out_tokens[(size_t)b * N + depth] = tok[next];
      ++depth;
      cur = next;
    }
    if (invalid) {
      st |= invalid == 4 ? ORC_ST_BAD_PARENT : ORC_ST_NONFINITE;
      for (int i = 0; i < N; ++i) {
        out_nodes[(size_t)b * N + i] = -1;
        out_tokens[(size_t)b * N + i] = -1;
      }
      n_acc[b] = -1;
      prob = 0.0;
      mg = mc = INFINITY;
      lo = hi = -1;
    } else {
      n_acc[b] = depth;
      out_tokens[(size_t)b * N + depth] = t;
    }
    out_prob[b] = prob;
    margin_acc[b] = (T == 0.0) ? INFINITY : mg;
    margin_cdf[b] = (T == 0.0) ? INFINITY : mc;
    cdf_lo[b] = lo;
    cdf_hi[b] = hi;
    put_tests(acc_tests, acc_flagged, b, T == 0.0 || invalid, nt, nf);
    status[b] = st;
  }
  free(p); free(q);
  return 0;
}

/* ------------------------------------------------------------------------
 * Geometric fan-out schedule (Saguaro, Theorem 12): w_k = a^{k/(1+r)} for
 * k < K, w_K = a^{K/(1+r)} (1-a)^{-1/(1+r)}, F_0 = budget / sum w, then the
 * real F_0 w_k made integer by largest remainder (ties to the lower k).
 * Returns nonzero on bad arguments.
 * ---------------------------------------------------------------------- */
int orc_fanout_schedule(int K, int budget, double a, double r, int32_t *F) {
  if (K < 0 || budget < 0 || !(a > 0.0 && a < 1.0) || !(r > 0.0)) return 1;
  double *w = malloc(sizeof(double) * (size_t)(K + 1));
  double *frac = malloc(sizeof(double) * (size_t)(K + 1));
  if (!w || !frac) { free(w); free(frac); return 1; }
  double s = 0.0;
  for (int k = 0; k < K; ++k) {
    w[k] = pow(a, (double)k / (1.0 + r));
    s += w[k];
  }
  w[K] = pow(a, (double)K / (1.0 + r)) * pow(1.0 - a, -1.0 / (1.0 + r));
  s += w[K];
  double F0 = (double)budget / s;
  int used = 0;
  for (int k = 0; k <= K; ++k) {
    double real = F0 * w[k];
    double fl = floor(real);
    F[k] = (int32_t)fl;
    frac[k] = real - fl;
    used += F[k];
  }
  for (int left = budget - used; left > 0; --left) {
    int best = -1;
    for (int k = 0; k <= K; ++k)
      if (frac[k] >= 0.0 && (best < 0 || frac[k] > frac[best])) best = k;
    if (best < 0) break;
    F[best] += 1;
    frac[best] = -1.0;
  }
  free(w); free(frac);
  return 0;
}

typedef struct { double v; int idx; } orc_entry;

static int entry_cmp(const void *x, const void *y) {
  const orc_entry *a = x, *b = y;
  if (a->v > b->v) return -1;
  if (a->v < b->v) return 1;
  return (a->idx > b->idx) - (a->idx < b->idx);
}

/* Top-F_k tokens of lookahead row k of every sequence (Saguaro, "speculation
 * cache strategy": the cache holds the top-F_k draft tokens at each
 * lookahead position).  draft [B, K+1, V]; out_tokens / out_logit [B, sum F]
 * grouped by k at offset sum_{k' < k} F_{k'}, best first.  A row holding a
 * NaN yields -1 tokens and status bit 2. */
int orc_fanout_topk(const void *draft, int dtype, int B, int K, int V,
                    const int32_t *F, int32_t *out_tokens, double *out_logit,
                    int32_t *status) {
  int total = 0;
  for (int k = 0; k <= K; ++k) total += F[k];
  orc_entry *e = malloc(sizeof(orc_entry) * (size_t)V);
  if (!e) return 1;
  for (int b = 0; b < B; ++b) {
    int st = 0, off = 0;
    for (int k = 0; k <= K; ++k) {
      size_t row = ((size_t)b * (K + 1) + k) * (size_t)V;
      int bad = 0;
      for (int j = 0; j < V; ++j) {
        double z = logit_at(draft, dtype, row + (size_t)j);
        if (isnan(z)) bad = 1;
        e[j].v = (z == 0.0) ? 0.0 : z; /* -0 and +0 are the same value */
        e[j].idx = j;
      }
      if (bad) st |= ORC_ST_NONFINITE;
      else qsort(e, (size_t)V, sizeof(orc_entry), entry_cmp);
      for (int i = 0; i < F[k]; ++i) {
        size_t o = (size_t)b * total + off + i;
        int ok = !bad && i < V;
        out_tokens[o] = ok ? e[i].idx : -1;
        if (out_logit) out_logit[o] = ok ? e[i].v : NAN;
      }
      off += F[k];
    }
    status[b] = st;
  }
  free(e);
  return 0;
}

/*
 * Cache hit of each sequence's verification outcome (Speculative Speculative
 * Decoding / Saguaro: the outcome is v = (k, t*), k accepted drafts and the
 * correction or bonus token t*; the cache holds, for each lookahead
 * position k, the F_k tokens of the fan-out row k).  hit[b] = 1 if t* is
 * one of the F_{n_b} tokens stored for position n_b, 0 if not, -1 for a
 * sequence without an outcome (n_b < 0).  tokens [B, K+1] (x_0..x_{n-1},
 * t*, ...), fan_tokens [B, sum F] grouped by position.
 */
int orc_fanout_hits(const int32_t *n_acc, const int32_t *tokens,
                    const int32_t *fan_tokens, const int32_t *F, int B,
                    int K, int32_t *hit) {
  int total = 0;
  for (int k = 0; k <= K; ++k) total += F[k];
  for (int b = 0; b < B; ++b) {
    const int n = n_acc[b];
    if (n < 0 || n > K) {
      hit[b] = -1;
      continue;
    }
    const int32_t t = tokens[(size_t)b * (K + 1) + n];
    int off = 0;
    for (int k = 0; k < n; ++k) off += F[k];
    int found = 0;
    for (int i = 0; i < F[n]; ++i)
      if (fan_tokens[(size_t)b * total + off + i] == t) found = 1;
    hit[b] = found;
  }
  return 0;
}

/* ------------------------------------------------------------------------
 * Filtered sampling of one row ("01 · Draft-then-verify", section 4,
 * standardised sampling): p = softmax(z / T); keep the top_k tokens in
 * (logit desc, index asc) order; of those, keep the smallest prefix whose
 * mass, renormalised over the top_k, reaches top_p (token i stays iff the
 * mass before it is below top_p); renormalise over the kept tokens.  p gets
 * the filtered distribution (0 outside the kept set).  *margin is lowered to
 * the distance of every prefix mass from top_p (where an fp32 computation
 * may cut the nucleus differently).  The kept count is written to *keep;
 * *keep_lo / *keep_hi (nullable) get the range of kept counts whose cut
 * lies within ORC_BAND of top_p (the counts an fp32 computation may reach:
 * a token whose renormalised prefix mass is below top_p - ORC_BAND stays in
 * every such count, one at or above top_p + ORC_BAND in none).  When
 * forced >= 1 the nucleus keeps that many tokens instead (at most top_k).
 * Returns 0 on an unusable row. */
static int filtered_row(const void *base, int dtype, size_t off, int V,
                        double T, int top_k, double top_p, double *p,
                        orc_entry *e, double *margin, int forced, int *keep_out,
                        int *keep_lo, int *keep_hi) {
  if (!softmax_row(base, dtype, off, V, T, p)) return 0;
  for (int j = 0; j < V; ++j) {
    double z = logit_at(base, dtype, off + (size_t)j);
    e[j].v = (z == 0.0) ? 0.0 : z;
    e[j].idx = j;
  }
  qsort(e, (size_t)V, sizeof(orc_entry), entry_cmp);
  int k = top_k < V ? top_k : V;
  double mk = 0.0;
  for (int i = 0; i < k; ++i) mk += p[e[i].idx];
  int keep = k, lo = k, hi = k;
  if (top_p < 1.0) {
    double before = 0.0;
    keep = lo = hi = 0;
    for (int i = 0; i < k; ++i) {
      double f = before / mk;
      note_margin(margin, fabs(f - top_p));
      if (f < top_p) keep = i + 1;
      if (f < top_p - ORC_BAND) lo = i + 1;
      if (f < top_p + ORC_BAND) hi = i + 1;
      before += p[e[i].idx];
    }
  }
  if (forced >= 1) keep = forced < k ? forced : k;
  *keep_out = keep;
  if (keep_lo) *keep_lo = lo;
  if (keep_hi) *keep_hi = hi;
  double S = 0.0;
  for (int i = 0; i < keep; ++i) S += p[e[i].idx];
  double *kept = malloc(sizeof(double) * (size_t)keep);
  if (!kept) return 0;
  for (int i = 0; i < keep; ++i) kept[i] = p[e[i].idx] / S;
  for (int j = 0; j < V; ++j) p[j] = 0.0;
  for (int i = 0; i < keep; ++i) p[e[i].idx] = kept[i];
  free(kept);
  return 1;
}

/* ------------------------------------------------------------------------
 * Linear verify with filtered sampling: the rule of orc_verify_linear with
 * p_i and q_i replaced by their top_k / top_p filtered versions (same
 * filter for target and draft).  T == 0 is greedy (the filters keep the
 * argmax), as in orc_verify_linear.  margin_acc also covers the nucleus
 * cuts (see filtered_row).
 * ---------------------------------------------------------------------- */
int orc_verify_linear_filtered(const void *target, const void *draft,
                               int dtype, const int32_t *tokens,
                               const float *uniforms, int B, int gamma, int V,
                               double T, int top_k, double top_p,
                               int32_t *n_acc, int32_t *out_tokens,
                               double *out_prob, double *margin_acc,
                               double *margin_cdf, int32_t *cdf_lo,
                               int32_t *cdf_hi, int32_t *acc_tests,
                               int32_t *acc_flagged, const int32_t *keep_forced,
                               int32_t *keep, int32_t *keep_lo,
                               int32_t *keep_hi, int32_t *status) {
  if (gamma > SD_ORC_MAX_GAMMA) return 1;
  if (T == 0.0) {
    double *acc = malloc(sizeof(double) * (size_t)(B * (gamma > 0 ? gamma : 1)));
    if (!acc) return 1;
    int rc = orc_verify_linear(target, draft, dtype, tokens, uniforms, B,
                               gamma, V, T, n_acc, out_tokens, out_prob, acc,
                               margin_acc, margin_cdf, cdf_lo, cdf_hi,
                               acc_tests, acc_flagged, NULL, status);
    free(acc);
    /* greedy: the filters keep the argmax; target rows 0..n are read (one
     * token kept each), draft rows are not */
    for (int b = 0; b < B && (keep || keep_lo || keep_hi); ++b)
      for (int i = 0; i < 2 * gamma + 1; ++i) {
        const int32_t v = (n_acc[b] >= 0 && i <= n_acc[b]) ? 1 : -1;
        if (keep) keep[(size_t)b * (2 * gamma + 1) + i] = v;
        if (keep_lo) keep_lo[(size_t)b * (2 * gamma + 1) + i] = v;
        if (keep_hi) keep_hi[(size_t)b * (2 * gamma + 1) + i] = v;
      }
    return rc;
  }
  double *p = malloc(sizeof(double) * (size_t)V);
  double *q = malloc(sizeof(double) * (size_t)V);
  double *w = malloc(sizeof(double) * (size_t)V);
  orc_entry *e = malloc(sizeof(orc_entry) * (size_t)V);
  if (!p || !q || !w || !e) { free(p); free(q); free(w); free(e); return 1; }
  const int G1 = gamma + 1, NS = 2 * gamma + 1;
  for (int b = 0; b < B; ++b) {
    int st = 0, n = 0, t = -1, invalid = 0, lo = -1, hi = -1, rejected = 0;
    int nt = 0, nf = 0;
    double mg = INFINITY, mc = INFINITY, mn = INFINITY, prob = 0.0;
    /* per-row kept counts: slot i for target row i, gamma + 1 + i for draft
     * row i; -1 for rows not read */
    int32_t kk[2 * SD_ORC_MAX_GAMMA + 1], klo[2 * SD_ORC_MAX_GAMMA + 1],
        khi[2 * SD_ORC_MAX_GAMMA + 1];
    for (int i = 0; i < NS; ++i) kk[i] = klo[i] = khi[i] = -1;
    const int32_t *fk = keep_forced ? keep_forced + (size_t)b * NS : NULL;
#define FROW(base, off, slot, dst)                                         \
  filtered_row(base, dtype, off, V, T, top_k, top_p, dst, e, &mn,          \
               fk ? fk[slot] : -1, &kk[slot], &klo[slot], &khi[slot])
    for (int i = 0; i < gamma; ++i) {
      if (!FROW(target, ((size_t)b * G1 + i) * V, i, p) ||
          !FROW(draft, ((size_t)b * gamma + i) * V, G1 + i, q)) {
        invalid = 1;
        break;
      }
      int x = tokens[(size_t)b * gamma + i];
      double r = (double)uniforms[(size_t)b * G1 + i];
      int ok;
      if (x < 0 || x >= V) {
        st |= ORC_ST_BAD_TOKEN;
        ok = 0;
      } else {
        double rho = accept_ratio(p[x], q[x]);
        note_test(&mg, &nt, &nf, r, rho);
        ok = (r <= rho);
      }
      if (!ok) { rejected = 1; break; }
      ++n;
    }
    if (!invalid) {
      if (rejected) { /* residual norm(max(0, p~_n - q~_n)) */
        double N = 0.0;
        for (int j = 0; j < V; ++j) {
          double d = p[j] - q[j];
          w[j] = d > 0.0 ? d : 0.0;
          N += w[j];
        }
        if (N == 0.0) {
          st |= ORC_ST_ZERO_MASS;
          for (int j = 0; j < V; ++j) w[j] = p[j];
        }
      } else if (!FROW(target, ((size_t)b * G1 + gamma) * V, gamma, p)) {
        invalid = 1;
      } else {
        for (int j = 0; j < V; ++j) w[j] = p[j];
      }
    }
    if (!invalid) {
      double u = (double)uniforms[(size_t)b * G1 + gamma];
      t = sample_icdf(w, V, u, &prob, &mc, &lo, &hi);
    } else {
      st |= ORC_ST_NONFINITE;
      n = -1;
      prob = 0.0;
      mg = mc = INFINITY;
      lo = hi = -1;
    }
    n_acc[b] = n;
    for (int i = 0; i < G1; ++i) {
      int32_t v = -1;
      if (!invalid) {
        if (i < n) v = tokens[(size_t)b * gamma + i];
        else if (i == n) v = t;
      }
      out_tokens[(size_t)b * G1 + i] = v;
    }
#undef FROW
    out_prob[b] = prob;
    /* the nucleus cuts count as flagged decisions unless the caller takes
     * their admissible ranges instead */
    margin_acc[b] = (keep_lo || mn > mg) ? mg : mn;
    margin_cdf[b] = mc;
    cdf_lo[b] = lo;
    cdf_hi[b] = hi;
    put_tests(acc_tests, acc_flagged, b, invalid, nt, nf);
    for (int i = 0; i < NS; ++i) {
      if (keep) keep[(size_t)b * NS + i] = invalid ? -1 : kk[i];
      if (keep_lo) keep_lo[(size_t)b * NS + i] = invalid ? -1 : klo[i];
      if (keep_hi) keep_hi[(size_t)b * NS + i] = invalid ? -1 : khi[i];
    }
    status[b] = st;
  }
  free(p); free(q); free(w); free(e);
  return 0;
}

/* ------------------------------------------------------------------------
 * Tree verify with deterministic drafts (SpecDiff-2, "greedy acceptance":
 * each drafted token is accepted with the verifier's probability of it,
 * independently of the drafter; on rejection the token is resampled from
 * the verifier's residual).  This is the tree rule above with the draft
 * distribution of child v replaced by the point mass on t_v: the ratio
 * p(t_v)/1 is p(t_v), and norm(max(0, p - delta_{t_v})) is p with t_v
 * removed and renormalised.  Arguments as orc_verify_tree, without draft.
 * A child whose token was removed already has p(t_v) = 0.  A token out of
 * range is rejected and removes nothing.
 * ---------------------------------------------------------------------- */
int orc_verify_tree_det(const void *target, int dtype, const int32_t *parent,
                        const int32_t *node_tokens, const float *uniforms,
                        int B, int N, int V, double T, int32_t *n_acc,
                        int32_t *out_tokens, int32_t *out_nodes,
                        double *out_prob, double *margin_acc,
                        double *margin_cdf, int32_t *cdf_lo, int32_t *cdf_hi,
                        int32_t *acc_tests, int32_t *acc_flagged,
                        int32_t *status) {
  double *p = malloc(sizeof(double) * (size_t)V);
  if (!p) return 1;
  for (int b = 0; b < B; ++b) {
    const int32_t *par = parent + (size_t)b * N;
    const int32_t *tok = node_tokens + (size_t)b * N;
    const float *U = uniforms + (size_t)b * N;
    int st = 0, invalid = 0, depth = 0, t = -1, lo = -1, hi = -1;
    int nt = 0, nf = 0;
    double mg = INFINITY, mc = INFINITY, prob = 0.0;
    for (int i = 0; i < N; ++i) {
      out_nodes[(size_t)b * N + i] = -1;
      out_tokens[(size_t)b * N + i] = -1;
    }
    if (par[0] != -1) invalid = 4;
    for (int v = 1; v < N && !invalid; ++v)
      if (par[v] < 0 || par[v] >= v) invalid = 4;
    int cur = 0;
    while (!invalid) {
      size_t off = ((size_t)b * N + cur) * (size_t)V;
      int next = -1;
      if (T == 0.0) {
        int a = argmax_row(target, dtype, off, V);
        if (a < 0) { invalid = 2; break; }
        for (int v = cur + 1; v < N; ++v) {
          if (par[v] != cur) continue;
          if (tok[v] < 0 || tok[v] >= V) st |= ORC_ST_BAD_TOKEN;
          if (tok[v] == a) { next = v; break; }
        }
        if (next < 0) { t = a; prob = 1.0; lo = hi = a; break; }
      } else {
        if (!softmax_row(target, dtype, off, V, T, p)) { invalid = 2; break; }
        int zero_mass = 0;
        for (int v = cur + 1; v < N && !zero_mass; ++v) {
          if (par[v] != cur) continue;
          int x = tok[v];
          if (x < 0 || x >= V) { st |= ORC_ST_BAD_TOKEN; continue; }
          double rho = p[x];
          note_test(&mg, &nt, &nf, (double)U[v], rho);
          if ((double)U[v] <= rho) { next = v; break; }
          /* rejected: remove x and renormalise */
          p[x] = 0.0;
          double S = 0.0;
          for (int j = 0; j < V; ++j) S += p[j];
          if (S == 0.0) {
            st |= ORC_ST_ZERO_MASS;
            softmax_row(target, dtype, off, V, T, p);
            zero_mass = 1;
          } else {
            for (int j = 0; j < V; ++j) p[j] /= S;
          }
        }
        if (next < 0) {
          t = sample_icdf(p, V, (double)U[0], &prob, &mc, &lo, &hi);
          break;
        }
      }
      out_nodes[(size_t)b * N + depth] = next;
      out_tokens[(size_t)b * N + depth] = tok[next];
      ++depth;
      cur = next;
    }
    if (invalid) {
      st |= invalid == 4 ? ORC_ST_BAD_PARENT : ORC_ST_NONFINITE;
      for (int i = 0; i < N; ++i) {
        out_nodes[(size_t)b * N + i] = -1;
        out_tokens[(size_t)b * N + i] = -1;
      }
      n_acc[b] = -1;
      prob = 0.0;
      mg = mc = INFINITY;
      lo = hi = -1;
    } else {
      n_acc[b] = depth;
      out_tokens[(size_t)b * N + depth] = t;
    }
    out_prob[b] = prob;
    margin_acc[b] = (T == 0.0) ? INFINITY : mg;
    margin_cdf[b] = (T == 0.0) ? INFINITY : mc;
    cdf_lo[b] = lo;
    cdf_hi[b] = hi;
    put_tests(acc_tests, acc_flagged, b, T == 0.0 || invalid, nt, nf);
    status[b] = st;
  }
  free(p);
  return 0;
}

/* ------------------------------------------------------------------------
 * K candidates verified as one token tree (the multi-draft reading of
 * SpecDiff-2's K iid candidates from shared position-wise marginals, with
 * PRESTO section 2.1's prefix-wise tree verification).  Candidate k's
 * token at position j (tokens [B, K, gamma]) is one node, N = 1 + K gamma
 * nodes per sequence, created position by position and, within a
 * position, in increasing k:
 *  - its parent is the node of candidate k's prefix (the root for j = 0);
 *  - if an earlier candidate with the same prefix has the same token at j,
 *    the node is a leaf duplicate (a repeated iid draw, kept so that the
 *    sibling rule sees every draw) and candidate k continues below the
 *    earlier candidate's node;
 *  - otherwise it is the node of the prefix through position j, with
 *    target row (k, j + 1) and draft row j + 1 (none at j + 1 == gamma).
 * The root has target row (0, 0) and draft row 0.  A duplicate copies the
 * rows of the node it repeats.  Node (k, j) tests with uniforms[b][k][j];
 * the final draw (tree slot 0) uses uniforms[b][0][gamma].  node_cand is
 * the candidate that created the node (the lowest k through a non-duplicate
 * node).  Row indices: target_row into the K (gamma + 1) rows of sequence
 * b (k (gamma + 1) + j), draft_row into its gamma rows, -1 for none.
 * ---------------------------------------------------------------------- */
int orc_kcand_trie(const int32_t *tokens, const float *uniforms, int B, int K,
                   int gamma, int32_t *parent, int32_t *node_tokens,
                   float *node_uniforms, int32_t *target_row,
                   int32_t *draft_row, int32_t *node_cand, int32_t *is_dup) {
  const int N = 1 + K * gamma, G1 = gamma + 1;
  int *at = malloc(sizeof(int) * (size_t)(K > 0 ? K : 1));
  if (!at) return 1;
  for (int b = 0; b < B; ++b) {
    int32_t *par = parent + (size_t)b * N, *tok = node_tokens + (size_t)b * N;
    float *U = node_uniforms + (size_t)b * N;
    int32_t *tr = target_row + (size_t)b * N, *dr = draft_row + (size_t)b * N;
    int32_t *nc = node_cand + (size_t)b * N, *dup = is_dup + (size_t)b * N;
    const int32_t *x = tokens + (size_t)b * K * gamma;
    const float *u = uniforms + (size_t)b * K * G1;
    par[0] = -1;
    tok[0] = -1;
    U[0] = u[gamma]; /* candidate 0, slot gamma */
    tr[0] = 0;
    dr[0] = gamma > 0 ? 0 : -1;
    nc[0] = 0;
    dup[0] = 0;
    for (int k = 0; k < K; ++k) at[k] = 0;
    int v = 1;
    for (int j = 0; j < gamma; ++j) {
      const int first = v; /* nodes of position j start here */
      for (int k = 0; k < K; ++k, ++v) {
        const int t = x[(size_t)k * gamma + j];
        int same = -1; /* an earlier non-duplicate node: same parent, token */
        for (int w = first; w < v && same < 0; ++w)
          if (!dup[w] && par[w] == at[k] && tok[w] == t) same = w;
        par[v] = at[k];
        tok[v] = t;
        U[v] = u[(size_t)k * G1 + j];
        nc[v] = k;
        if (same >= 0) {
          dup[v] = 1;
          tr[v] = tr[same];
          dr[v] = dr[same];
          at[k] = same;
        } else {
          dup[v] = 0;
          tr[v] = k * G1 + j + 1;
          dr[v] = j + 1 < gamma ? j + 1 : -1;
          at[k] = v;
        }
      }
    }
  }
  free(at);
  return 0;
}

/* ------------------------------------------------------------------------
 * PRESTO tree construction, one depth ("PRESTO", section 4.1: the
 * prefix-aligned score s_{d,t}(c_d) = log q_d(t) + lambda_d log rho_d(t |
 * c_d) and the path score S(P), Eq. 10, the sum of s along the path;
 * section 4.2 and its Algorithm 1: beam search with global retention under
 * a node budget).  One call expands depth d of every sequence's tree:
 *  - the frontier holds up to W paths (frontier_node[b][w] >= 0, their
 *    path scores frontier_score[b][w]); path w's prefix signal is the row
 *    log_rho[b][w] (log rho, <= 0; -inf for rho = 0);
 *  - path w proposes its b_top tokens of largest s (ties to the lower id),
 *    tokens with s = -inf excluded, each with candidate score S_w + s;
 *  - all candidates of the sequence are ordered by (score desc, w asc,
 *    token asc) and the first min(count, budget - n_nodes) become nodes
 *    n_nodes, n_nodes + 1, ... (parent: the path's node);
 *  - the new frontier is the first min(W, added) of them, in that order.
 * log q_d is log softmax(z / T) of the drafter's marginal row q_logits[b]
 * (row stride q_stride elements).  A NaN or +inf in a row read makes the
 * sequence invalid: n_nodes = -1, frontier cleared (status 2).  margin[b]
 * is the smallest nonzero score gap that decided the outcome: at each
 * path's top-b cut, and between consecutive candidates of the merged order
 * up to one past the last added (INFINITY when nothing was decided).
 * Exact ties (equal inputs, e.g. repeated bf16 logits) are decided by the
 * stated order, not by rounding, so they set no margin.
 * ---------------------------------------------------------------------- */
#define SD_ORC_MAX_W 64
typedef struct { double s; int w, tok; } orc_cand;

static int cand_cmp(const void *x, const void *y) {
  const orc_cand *a = x, *b = y;
  if (a->s != b->s) return a->s < b->s ? 1 : -1;
  if (a->w != b->w) return a->w - b->w;
  return a->tok - b->tok;
}

int orc_presto_expand(const void *q_logits, const void *log_rho, int dtype,
                      long long q_stride, int B, int W, int V, double T,
                      double lambda, int b_top, int budget, int32_t *n_nodes,
                      int32_t *parent, int32_t *node_tokens,
                      double *node_score, int32_t *frontier_node,
                      double *frontier_score, double *margin,
                      int32_t *status) {
  if (W < 1 || W > SD_ORC_MAX_W || b_top < 1 || budget < 1 || lambda < 0.0)
    return 1;
  orc_cand *row = malloc(sizeof(orc_cand) * (size_t)V);
  orc_cand *all = malloc(sizeof(orc_cand) * (size_t)(W * b_top + 1));
  double *lq = malloc(sizeof(double) * (size_t)V);
  if (!row || !all || !lq) { free(row); free(all); free(lq); return 1; }
  for (int b = 0; b < B; ++b) {
    int32_t *fn = frontier_node + (size_t)b * W;
    double *fs = frontier_score + (size_t)b * W;
    double mg = INFINITY;
    int st = 0;
    const int n0 = n_nodes[b];
    if (n0 < 0 || n0 >= budget) { margin[b] = mg; status[b] = 0; continue; }
    const size_t qoff = (size_t)b * (size_t)q_stride;
    int invalid = !softmax_row(q_logits, dtype, qoff, V, T, lq);
    for (int j = 0; j < V && !invalid; ++j) lq[j] = log(lq[j]);
    int nc = 0;
    for (int w = 0; w < W && !invalid; ++w) {
      if (fn[w] < 0) continue;
      const size_t roff = ((size_t)b * W + w) * (size_t)V;
      for (int j = 0; j < V; ++j) {
        /* lambda == 0: the prefix signal is not used (nor read);
         * lambda * (-inf) is -inf for lambda > 0 */
        double r = lambda == 0.0 ? 0.0 : logit_at(log_rho, dtype,
                                                  roff + (size_t)j);
        if (isnan(r) || r == INFINITY) { invalid = 1; break; }
        double s = lq[j] + (lambda == 0.0 ? 0.0 : lambda * r);
        row[j].s = s;
        row[j].w = w;
        row[j].tok = j;
      }
      if (invalid) break;
      qsort(row, (size_t)V, sizeof(orc_cand), cand_cmp);
      int take = 0;
      while (take < b_top && take < V && row[take].s > -INFINITY) ++take;
      if (take == b_top && take < V && row[take].s > -INFINITY &&
          row[take - 1].s != row[take].s)
        note_margin(&mg, row[take - 1].s - row[take].s);
      for (int i = 0; i < take; ++i) {
        all[nc] = row[i];
        all[nc].s = fs[w] + row[i].s;
        ++nc;
      }
    }
    if (invalid) {
      n_nodes[b] = -1;
      for (int w = 0; w < W; ++w) { fn[w] = -1; fs[w] = 0.0; }
      margin[b] = INFINITY;
      status[b] = ORC_ST_NONFINITE;
      continue;
    }
    qsort(all, (size_t)nc, sizeof(orc_cand), cand_cmp);
    int add = budget - n0 < nc ? budget - n0 : nc;
    for (int i = 0; i + 1 < nc && i < add; ++i)
      if (all[i].s != all[i + 1].s) note_margin(&mg, all[i].s - all[i + 1].s);
    int32_t old_fn[SD_ORC_MAX_W];
    for (int w = 0; w < W; ++w) old_fn[w] = fn[w];
    for (int i = 0; i < add; ++i) {
      const size_t v = (size_t)b * budget + (size_t)(n0 + i);
      parent[v] = old_fn[all[i].w];
      node_tokens[v] = all[i].tok;
      node_score[v] = all[i].s;
    }
    for (int w = 0; w < W; ++w) {
      fn[w] = w < add ? n0 + w : -1;
      fs[w] = w < add ? all[w].s : 0.0;
    }
    n_nodes[b] = n0 + add;
    margin[b] = mg;
    status[b] = st;
  }
  free(row); free(all); free(lq);
  return 0;
}

/* ------------------------------------------------------------------------
 * SpecBranch branch resampling ("SpecBranch", branch resampling: at the
 * branch point x_b fork k = max(1, floor(k_max (1 - q(x_b)))) parallel
 * branches, the Top-k of the draft distribution there).  q = softmax(z / T)
 * of draft row b (T == 0: the point mass on the argmax); q(x_b) is the
 * drafted token's probability.  k is capped at V.  out_tokens [B, k_max]:
 * the k tokens of largest logit (ties to the lower id), then -1.
 * margin[b]: relative distance of k_max q(x_b) to the nearest integer at
 * which k = max(1, min(V, k_max - ceil(k_max q))) steps (a finite-
 * precision q could go either way there); INFINITY at T == 0 or when k
 * cannot step.
 * An x_b outside [0, V) or an unusable row: k = -1, tokens -1, status.
 * ---------------------------------------------------------------------- */
int orc_branch_fork(const void *draft, int dtype, const int32_t *x_b, int B,
                    int V, double T, int k_max, int32_t *out_k,
                    int32_t *out_tokens, double *margin, int32_t *status) {
  if (k_max < 1) return 1;
  double *q = malloc(sizeof(double) * (size_t)V);
  orc_entry *e = malloc(sizeof(orc_entry) * (size_t)V);
  if (!q || !e) { free(q); free(e); return 1; }
  for (int b = 0; b < B; ++b) {
    const size_t off = (size_t)b * V;
    int32_t *ot = out_tokens + (size_t)b * k_max;
    for (int i = 0; i < k_max; ++i) ot[i] = -1;
    margin[b] = INFINITY;
    status[b] = 0;
    out_k[b] = -1;
    const int x = x_b[b];
    double qx;
    if (T == 0.0) {
      int a = argmax_row(draft, dtype, off, V);
      if (a < 0) { status[b] = ORC_ST_NONFINITE; continue; }
      qx = (x == a) ? 1.0 : 0.0;
    } else {
      if (!softmax_row(draft, dtype, off, V, T, q)) {
        status[b] = ORC_ST_NONFINITE;
        continue;
      }
      qx = (x >= 0 && x < V) ? q[x] : 0.0;
    }
    if (x < 0 || x >= V) { status[b] = ORC_ST_BAD_TOKEN; continue; }
    /* floor(k_max (1 - q)) written as k_max - ceil(k_max q): the same
     * integer, without 1 - q rounding to 1 when q is tiny */
    const double y = (double)k_max * qx;
    int k = k_max - (int)ceil(y);
    if (k < 1) k = 1;
    if (k > V) k = V;
    if (T != 0.0) {
      /* relative distance of y to the nearest integer n at which the
       * clamped k steps (ceil(y) going from n to n + 1 changes k: n in
       * [max(1, k_max - V), k_max - 2]); y below ~1e-30 could vanish in
       * finite precision */
      const double lo = k_max - V > 1 ? (double)(k_max - V) : 1.0;
      const double hi = (double)(k_max - 2);
      if (lo > hi) {
        margin[b] = INFINITY;
      } else {
        double n = floor(y + 0.5);
        if (n < lo) n = lo;
        if (n > hi) n = hi;
        margin[b] = y < 1e-30 ? 0.0 : fabs(y - n) / y;
      }
    }
    for (int j = 0; j < V; ++j) {
      e[j].v = logit_at(draft, dtype, off + (size_t)j);
      if (e[j].v == 0.0) e[j].v = 0.0; /* -0 equals +0 */
      e[j].idx = j;
    }
    qsort(e, (size_t)V, sizeof(orc_entry), entry_cmp);
    for (int i = 0; i < k; ++i) ot[i] = e[i].idx;
    out_k[b] = k;
  }
  free(q); free(e);
  return 0;
}
