/*
 * sd_verify.h -- C ABI of the GB300 (sm_103a) verify step of speculative
 * decoding ("draft-then-verify" at temperature T).
 *
 * What is computed (citations are to the pages this library implements):
 *
 *  - "01 · Draft-then-verify" (llm-infra-atlas), section 1, Algorithm 1 and
 *    section 4, the spec_step listing: for each sequence, with p_i the target
 *    distribution and q_i the draft distribution at position i, draw r_i and
 *    accept draft token x_i iff r_i <= p_i(x_i) / q_i(x_i), scanning left to
 *    right and stopping at the first rejection; a rejection at position n
 *    emits a correction drawn from norm(max(0, p_n - q_n)) (section 2.1);
 *    when all gamma drafts are accepted a bonus token is drawn from p_gamma
 *    (0-based).  Temperature reduces to sampling softmax(z / T) (section 1,
 *    notation); T == 0 is greedy: accept iff x_i == argmax p_i (section 2.2).
 *  - SpecDiff-2 (MLSys 2026), "core method", self-selection acceptance: K
 *    candidate drafts sampled from shared position-wise marginals; all are
 *    verified and the one with the longest accepted streak is kept.
 *  - PRESTO, section 2.1 (tree-based speculative decoding): a token tree is
 *    verified prefix-wise from the root; siblings are tried in turn with
 *    p <- norm(max(0, p - q)) after each rejection.
 *  - Speculative Speculative Decoding / Saguaro, "speculation cache
 *    strategy", Theorem 12: geometric fan-out F_k = F_0 a^{k/(1+r)} (k < K),
 *    F_K = F_0 a^{K/(1+r)} (1-a)^{-1/(1+r)}, sum F_k = budget; the cache holds
 *    the top-F_k draft tokens of each lookahead position k; "technical
 *    architecture": a verification outcome is served from the cache when it
 *    is in it.
 *  - SpecDiff-2, "core method", greedy acceptance: a drafted token accepted
 *    with the verifier's probability of it (deterministic drafts).
 *  - "01 · Draft-then-verify", section 4 (standardised sampling): top-k and
 *    nucleus filtering act on p and q before the ratio.
 *  - PRESTO, sections 4.1-4.4: tree construction with the prefix-aligned
 *    score log q + lambda log rho (a product of experts) under a node budget.
 *  - SpecBranch, branch resampling: k = max(1, floor(k_max (1 - q(x_b))))
 *    top-k branches at a branch point.
 *
 * Entry points: sd_verify_linear (and _static, _filtered), sd_verify_kcand,
 * sd_verify_kcand_trie, sd_verify_tree, sd_verify_tree_det,
 * sd_fanout_schedule (host), sd_fanout_topk, sd_fanout_hits,
 * sd_verify_linear_fanout, sd_presto_init, sd_presto_expand,
 * sd_branch_fork; each call with a workspace has a *_workspace query.
 *
 * Conventions shared by every call:
 *  - Every tensor argument is a DEVICE pointer owned by the caller, row-major
 *    and contiguous, unless marked "host".  The library never allocates,
 *    frees or synchronises inside a verify call; all work is enqueued on
 *    `stream` (a cudaStream_t; NULL is the legacy default stream).
 *  - Logits are fp32 (SD_F32) or bf16 (SD_BF16); all arithmetic is fp32.
 *  - Uniform numbers are inputs, each in (0, 1).
 *  - The return value reports host-side validation and launch errors only;
 *    it is SD_OK when the work was enqueued.  Problems found in the data
 *    are reported by OR-ing SD_DEV_* bits into *dev_status (nullable, a
 *    device int32 the caller zeroes) and by the per-sequence outputs
 *    described below.  Kernels never trap.
 *  - Workspace: a device buffer of at least the size the matching
 *    *_workspace() query returns (may be NULL when that size is 0).  It
 *    holds a work-queue counter that each call resets on its stream, so two
 *    calls that may overlap on the GPU must not share a workspace.
 *  - Only sm_103 devices are supported; other devices get
 *    SD_ERR_UNSUPPORTED.  There is no fallback path.
 *  - sd_last_error() returns a short thread-local text for the last failed
 *    call of this thread.
 */
#ifndef SD_VERIFY_H
#define SD_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SD_OK = 0,
  SD_ERR_INVALID_ARG = 1, /* null pointer, bad size, T < 0 or NaN, ... */
  SD_ERR_UNSUPPORTED = 2, /* not an sm_103 device, or a size beyond a limit */
  SD_ERR_CUDA = 3         /* a CUDA runtime call failed */
} sd_status;

typedef enum { SD_F32 = 0, SD_BF16 = 1 } sd_dtype;

/* device status bits */
#define SD_DEV_BAD_TOKEN 1  /* a draft token outside [0, V): that test rejects */
#define SD_DEV_NONFINITE 2  /* a row read held NaN or +inf, or only -inf:
                               the sequence's outputs are -1 */
#define SD_DEV_BAD_PARENT 4 /* tree: parent[0] != -1 or parent[v] not in
                               [0, v): the tree's outputs are -1 */
#define SD_DEV_ZERO_MASS 8  /* a residual had zero mass: drawn from p instead */
#define SD_DEV_TIMEOUT 16   /* a bounded wait on an asynchronous copy gave up:
                               the call's outputs are not to be trusted */

/* Limits (SD_ERR_UNSUPPORTED beyond them). */
#define SD_MAX_V (1 << 24)     /* vocabulary size */
#define SD_MAX_GAMMA 64        /* draft length (linear, kcand) */
#define SD_MAX_K 32            /* candidates (kcand); lookahead positions - 1 (fan-out) */
#define SD_MAX_TREE_NODES 1024 /* nodes per tree */
#define SD_MAX_FANOUT 64       /* F_k per position */

const char *sd_version(void);
const char *sd_last_error(void);

/* ---------------------------------------------------------------------
 * Tuning switches (no counterpart in the pages).  Each one picks among
 * kernels or launch shapes that compute the same results; the defaults are
 * the fastest measured on the workloads this library is tuned for.  They
 * are process-wide, read by the next call that launches work, and never
 * taken from the environment.  sd_tune_set returns SD_ERR_INVALID_ARG for
 * an unknown key or a value outside the key's range; sd_tune_get returns
 * the current value (-1 for an unknown key).  Not synchronised with calls
 * running on other host threads: set them before such calls start.
 * ------------------------------------------------------------------- */
typedef enum {
  SD_TUNE_CLUSTER = 0,         /* CTAs per cluster (linear, tree, fused,
                                  filtered, kcand): 0 chosen, 1/2/4/8/16 */
  SD_TUNE_NO_TMA = 1,          /* 1: plain 16-byte loads instead of the TMA
                                  ring (linear, tree); default 0 */
  SD_TUNE_ALLROWS = 2,         /* small linear inputs read every row in one
                                  launch: 0 never, 1 up to 64 MB (default),
                                  2 wherever its scratch fits */
  SD_TUNE_SPEC = 3,            /* a cluster's last sequence reads ahead: 0
                                  never, 1 (default), 2 also L2 prefetch */
  SD_TUNE_FUSED = 4,           /* sd_verify_linear_fanout: 1 one launch
                                  (default), 0 the two calls */
  SD_TUNE_KCAND_RING = 5,      /* 0: K-candidate verify without the TMA
                                  ring; default 1 */
  SD_TUNE_FANOUT_CLUSTER = 6,  /* fan-out CTAs per cluster: 0 chosen */
  SD_TUNE_FANOUT_LDG = 7,      /* 1: fan-out with plain loads; default 0 */
  SD_TUNE_FANOUT_MAXC = 8,     /* cap on the fan-out's clusters: 0 none */
  SD_TUNE_FANOUT_L2_FIRST = 9, /* fan-out rows read evict-first: default 1 */
  SD_TUNE_HELPERS = 10,        /* linear and K-candidate verify: clusters
                                  with no sequence left compute row
                                  statistics ahead of the scans still
                                  running: 0 or 1 (default 1) */
  SD_TUNE_COUNT = 11
} sd_tune;

sd_status sd_tune_set(sd_tune key, int value);
int sd_tune_get(sd_tune key);

/* ---------------------------------------------------------------------
 * Linear verify ("01 · Draft-then-verify", Algorithm 1 / spec_step).
 *
 * target_logits [B, gamma+1, V]: row i is the target logits p_i given the
 *     prefix and x_0..x_{i-1}; row gamma feeds the bonus draw.
 * draft_logits [B, gamma, V]: row i is the draft logits that produced
 *     x_i.  May be NULL when T == 0 (greedy reads no draft logits).
 * draft_tokens [B, gamma] int32.
 * uniforms [B, gamma+1] float: slot i < gamma is r_i of the accept test,
 *     slot gamma is the draw of the correction or bonus token.
 * T: temperature, >= 0 (0 = greedy).
 *
 * Outputs (device):
 *   n_accepted [B]: accepted drafts n in [0, gamma] (-1: invalid rows).
 *   out_tokens [B, gamma+1]: x_0..x_{n-1}, then the correction/bonus
 *       token, then -1 padding.
 *   out_prob [B] (nullable): probability of the last token under the
 *       distribution it was drawn from (1 when T == 0).
 *   out_accept_prob [B, gamma] (nullable): min(1, p_i(x_i)/q_i(x_i)) of
 *       each test made (1/0 when T == 0), -1 for positions after the first
 *       rejection (never tested: their logits are never read).
 *   out_resid [B, V] (nullable, debug): the normalised distribution the last
 *       token was drawn from (one-hot when T == 0).  Costs an extra pass.
 * The scan reads only the rows the method needs: target rows 0..n, draft
 * rows 0..min(n, gamma-1).  With SD_TUNE_HELPERS on (the default), clusters
 * that have no sequence left also read rows ahead of the scans still
 * running (rows of positions up to gamma), so that a scan finds them done;
 * the results are the same bits either way.
 * Workspace: sd_verify_linear_workspace(B, gamma, V, dt) bytes.  Which of
 * the two paths runs (every row's statistics in one launch, or one cluster
 * walk per sequence) depends on the sizes, the pointers' alignment and
 * SD_TUNE_ALLROWS only, never on scratch handed over beyond that figure.
 * ------------------------------------------------------------------- */
size_t sd_verify_linear_workspace(int B, int gamma, int V, sd_dtype dt);

sd_status sd_verify_linear(const void *target_logits, const void *draft_logits,
                           sd_dtype dt, const int32_t *draft_tokens,
                           const float *uniforms, int B, int gamma, int V,
                           float T, int32_t *n_accepted, int32_t *out_tokens,
                           float *out_prob, float *out_accept_prob,
                           float *out_resid, int32_t *dev_status,
                           void *workspace, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------
 * Linear verify without a caller workspace (no counterpart in the pages:
 * a deployment convenience for callers that must not allocate).
 *
 * Arguments and results as sd_verify_linear, minus workspace / ws_bytes.
 * The scratch is a file-scope device array of SD_STATIC_WS_BYTES per
 * device.  A call whose sd_verify_linear_workspace(B, gamma, V, dt)
 * exceeds it returns SD_ERR_UNSUPPORTED (nothing is launched).  The first
 * call on a device looks the array's address up (cudaGetSymbolAddress,
 * with that device current) and caches it: make that first call before
 * any stream capture.  The call allocates and frees nothing; it clears the
 * counters that must start at zero with a memset on `stream`.  Calls whose
 * work overlaps on the GPU (other streams, other host threads) share the
 * array and race: serialise them.
 * ------------------------------------------------------------------- */
#define SD_STATIC_WS_BYTES (1u << 20)

sd_status sd_verify_linear_static(
    const void *target_logits, const void *draft_logits, sd_dtype dt,
    const int32_t *draft_tokens, const float *uniforms, int B, int gamma,
    int V, float T, int32_t *n_accepted, int32_t *out_tokens, float *out_prob,
    float *out_accept_prob, float *out_resid, int32_t *dev_status,
    void *stream);

/* ---------------------------------------------------------------------
 * Linear verify with filtered sampling ("01 · Draft-then-verify", section
 * 4, standardised sampling: top-k / nucleus act on p and q before the
 * ratio is formed).
 *
 * Arguments and outputs as sd_verify_linear (no out_accept_prob /
 * out_resid), plus:
 *   top_k >= 1: keep the top_k tokens by (logit desc, id asc); top_k >= V
 *       keeps every token;
 *   top_p in (0, 1]: then keep the smallest prefix of them, in that order,
 *       whose mass renormalised over the top_k reaches top_p (a token stays
 *       iff the mass before it is below top_p; 1: all).
 *   out_keep [B, 2 gamma + 1] int32 (nullable, debug): the number of
 *       tokens each row read kept (slot i: target row i, slot gamma + 1 + i:
 *       draft row i; -1 for rows not read, or every slot of an unusable
 *       sequence).
 * p~ and q~ are softmax(z / T) restricted to the kept tokens and
 * renormalised; x_i is accepted iff r_i <= p~_i(x_i) / q~_i(x_i); the
 * correction is drawn from norm(max(0, p~_n - q~_n)), the bonus from
 * p~_gamma.  T == 0 is greedy (the filters keep the argmax), as in
 * sd_verify_linear.  Rows must be 16-byte aligned (V * elt a multiple of
 * 16), else SD_ERR_UNSUPPORTED.  Each row the method needs is read once.
 * With top_k <= SD_MAX_FANOUT the rows' exact top-k lists are kept in
 * registers; above it (or with top_k >= V) a cluster holds each row pair
 * in shared memory and selects the cut by histogram: V * elt may then be
 * at most about 1.6 MB (SD_ERR_UNSUPPORTED beyond).
 * ------------------------------------------------------------------- */
size_t sd_verify_linear_filtered_workspace(int B, int gamma, int V,
                                           sd_dtype dt);

sd_status sd_verify_linear_filtered(
    const void *target_logits, const void *draft_logits, sd_dtype dt,
    const int32_t *draft_tokens, const float *uniforms, int B, int gamma,
    int V, float T, int top_k, float top_p, int32_t *n_accepted,
    int32_t *out_tokens, float *out_prob, int32_t *out_keep,
    int32_t *dev_status, void *workspace, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------
 * K-candidate verify with verifier self-selection (SpecDiff-2, "core
 * method").
 *
 * target_logits [B, K, gamma+1, V]: candidate k's own target rows.
 * draft_logits [B, gamma, V]: the position-wise draft marginals shared by
 *     all K candidates.
 * draft_tokens [B, K, gamma]; uniforms [B, K, gamma+1] (slot [b][k][i] is
 *     the accept draw of candidate k at position i; [b][k*][gamma] is the
 *     final draw of the selected candidate).
 * Every candidate is verified with the linear rule; k* is the candidate
 * with the largest accepted count (lowest k on ties); the correction or
 * bonus token is drawn for k* only.
 * Outputs: n_accepted [B], selected_k [B], out_tokens [B, gamma+1],
 *   n_per_cand [B, K] (nullable), out_prob [B] (nullable).
 * This selection is not distribution-preserving for K > 1.
 * With SD_TUNE_HELPERS on (the default; sampled, aligned rows, K <= 31),
 * clusters whose sequence is done also read rows of positions ahead of the
 * scans still running; the results are the same bits either way.
 * Workspace: sd_verify_kcand_workspace bytes (the work counter and up to
 * 64 MB of helping records).
 * ------------------------------------------------------------------- */
size_t sd_verify_kcand_workspace(int B, int K, int gamma, int V, sd_dtype dt);

sd_status sd_verify_kcand(const void *target_logits, const void *draft_logits,
                          sd_dtype dt, const int32_t *draft_tokens,
                          const float *uniforms, int B, int K, int gamma,
                          int V, float T, int32_t *n_accepted,
                          int32_t *selected_k, int32_t *out_tokens,
                          int32_t *n_per_cand, float *out_prob,
                          int32_t *dev_status, void *workspace,
                          size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------
 * Token-tree verify (PRESTO section 2.1; sibling rule as stated above).
 *
 * target_logits [B, N, V]: row u is p(. | path to u).
 * draft_logits [B, N, V]: row u is the q that drafted u's children (rows
 *     of leaves are never read).
 * parent [B, N] int32: parent[0] = -1, 0 <= parent[v] < v.
 * node_tokens [B, N] int32: token of node v (slot 0 unused).
 * uniforms [B, N] float: slot v tests node v, slot 0 is the final draw.
 * From the root, the children of the current node are tried in increasing
 * node index, each against the current p and the parent's draft row q;
 * after a rejection p becomes norm(max(0, p - q)); an accepted child becomes
 * the current node.  When no child is accepted, or at a leaf, the last token
 * is drawn from the current p.
 * Outputs: n_accepted [B] (accepted depth), out_tokens [B, N] (accepted
 *   tokens then the final token, -1 padded), out_nodes [B, N] (accepted
 *   node ids, -1 padded), out_prob [B] (nullable).
 * ------------------------------------------------------------------- */
size_t sd_verify_tree_workspace(int B, int N, int V, sd_dtype dt);

sd_status sd_verify_tree(const void *target_logits, const void *draft_logits,
                         sd_dtype dt, const int32_t *parent,
                         const int32_t *node_tokens, const float *uniforms,
                         int B, int N, int V, float T, int32_t *n_accepted,
                         int32_t *out_tokens, int32_t *out_nodes,
                         float *out_prob, int32_t *dev_status,
                         void *workspace, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------
 * K candidate drafts verified as one token tree (SpecDiff-2, "core
 * method": K candidates drawn independently from the shared position-wise
 * marginals; PRESTO section 2.1: a token tree is verified prefix-wise from
 * the root).  Unlike sd_verify_kcand's self-selection, the output is
 * distributed as the target.
 *
 * Arguments as sd_verify_kcand (target_logits [B, K, gamma+1, V],
 * draft_logits [B, gamma, V], draft_tokens [B, K, gamma], uniforms
 * [B, K, gamma+1]), with K <= 32 and 1 + K gamma <= SD_MAX_TREE_NODES.
 * The tree: candidate k's token at position j is node 1 + j K + k, below
 * the node of its prefix (node 0, the root, for j = 0).  A token repeating
 * an earlier candidate's token under the same prefix is a leaf duplicate
 * and that candidate continues below the first copy; any other node reads
 * target row (k, j+1) and draft row j+1.  The root reads target row (0, 0)
 * and draft row 0.  The walk is sd_verify_tree's: node (k, j) tests with
 * uniforms[b][k][j], the final draw uses uniforms[b][0][gamma].
 * Outputs: n_accepted [B], out_tokens [B, gamma+1] (accepted tokens, the
 *   final token, -1 padding), selected_k [B] (nullable: the candidate that
 *   created the last accepted node, 0 when none was accepted, -1 for an
 *   invalid sequence), out_prob [B] (nullable).
 * Workspace: sd_verify_kcand_trie_workspace bytes (the tree, 24 B a node).
 * ------------------------------------------------------------------- */
size_t sd_verify_kcand_trie_workspace(int B, int K, int gamma, int V,
                                      sd_dtype dt);

sd_status sd_verify_kcand_trie(const void *target_logits,
                               const void *draft_logits, sd_dtype dt,
                               const int32_t *draft_tokens,
                               const float *uniforms, int B, int K,
                               int gamma, int V, float T,
                               int32_t *n_accepted, int32_t *selected_k,
                               int32_t *out_tokens, float *out_prob,
                               int32_t *dev_status, void *workspace,
                               size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------
 * Token-tree verify with deterministic drafts (SpecDiff-2, "core method",
 * greedy acceptance: each drafted token is accepted with the verifier's
 * probability of it, independently of the drafter, and a rejection is
 * resampled from the verifier's residual).  This is the tree rule of
 * sd_verify_tree with the draft distribution of every child the point mass
 * on its token: child v is accepted iff uniforms[b][v] <= p'(t_v), where
 * p' is softmax(target row / T) with the tokens of the rejected siblings
 * removed and renormalised; a child whose token was removed already has
 * p'(t_v) = 0; a token outside [0, V) is rejected, removes nothing and sets
 * SD_DEV_BAD_TOKEN.  When every child is rejected, or at a leaf, the last
 * token is drawn from p' by inverse CDF with uniforms[b][0].  Lossless for
 * any deterministic choice of children (top-k trees included).  T == 0 is
 * the greedy walk of sd_verify_tree.
 *
 * Arguments, layouts, outputs, ownership and errors as sd_verify_tree,
 * without draft_logits (no draft row is read).  A removed mass that leaves
 * nothing falls back to p and sets SD_DEV_ZERO_MASS.
 * ------------------------------------------------------------------- */
size_t sd_verify_tree_det_workspace(int B, int N, int V, sd_dtype dt);

sd_status sd_verify_tree_det(const void *target_logits, sd_dtype dt,
                             const int32_t *parent,
                             const int32_t *node_tokens,
                             const float *uniforms, int B, int N, int V,
                             float T, int32_t *n_accepted,
                             int32_t *out_tokens, int32_t *out_nodes,
                             float *out_prob, int32_t *dev_status,
                             void *workspace, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------
 * PRESTO tree construction, one depth per call ("PRESTO", section 4.1:
 * prefix-aligned score s_{d,t}(c_d) = log q_d(t) + lambda log rho_d(t |
 * c_d), path score S(P) (Eq. 10) the sum of s along the path; section 4.2
 * and Algorithm 1: beam search with global retention under a node budget;
 * section 4.4: s is the log of the product of experts q rho^lambda up to
 * a constant).  rho is given; its learned predictor is not part of this.
 *
 * Tree state (device, caller-owned, updated in place):
 *   n_nodes [B] (nodes so far; -1 for an invalid sequence), parent,
 *   node_tokens [B, budget] int32, node_score [B, budget] float (S of the
 *   node's path), frontier_node [B, W] (node of frontier path w, -1 for an
 *   empty slot), frontier_score [B, W].  sd_presto_init sets the root:
 *   node 0 (parent -1, token -1, score 0), the only frontier path.
 * One depth: q_logits row b (at q_logits + b q_stride elements, q_stride
 *   >= V, so a [B, D, V] tensor's depth d is passed without a copy) is the
 *   drafter's marginal at this depth, log q_d = log softmax(z / T);
 *   log_rho [B, W, V] (not read when lambda == 0): log rho of frontier path
 *   w's prefix (<= 0, -inf for rho = 0).  Path w proposes its b_top tokens
 *   of largest s (ties to the lower id; s = -inf never), each with score
 *   S_w + s.  The proposals of a sequence are ordered by (score desc, w
 *   asc, token asc); the first min(count, budget - n_nodes) become nodes
 *   n_nodes, n_nodes + 1, ... in that order; the first min(W, added) of
 *   them are the new frontier (the other slots -1).  A sequence with
 *   n_nodes >= budget or < 0 is left as is.  A NaN or +inf in a row read
 *   makes the sequence invalid: n_nodes = -1, frontier cleared,
 *   SD_DEV_NONFINITE.  Requires T > 0, lambda >= 0, 1 <= W, b_top <= 64,
 *   W b_top <= 1024.  Scores are fp32.
 * ------------------------------------------------------------------- */
sd_status sd_presto_init(int B, int W, int budget, int32_t *n_nodes,
                         int32_t *parent, int32_t *node_tokens,
                         float *node_score, int32_t *frontier_node,
                         float *frontier_score, void *stream);

size_t sd_presto_expand_workspace(int B, int W, int V, int b_top,
                                  sd_dtype dt);

sd_status sd_presto_expand(const void *q_logits, long long q_stride,
                           const void *log_rho, sd_dtype dt, int B, int W,
                           int V, float T, float lambda, int b_top,
                           int budget, int32_t *n_nodes, int32_t *parent,
                           int32_t *node_tokens, float *node_score,
                           int32_t *frontier_node, float *frontier_score,
                           int32_t *dev_status, void *workspace,
                           size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------
 * SpecBranch branch resampling ("SpecBranch", branch resampling: at the
 * branch point x_b fork k = max(1, floor(k_max (1 - q(x_b)))) parallel
 * branches, the Top-k of the draft distribution there).
 *
 * draft_logits [B, V]: the draft row at each sequence's branch point;
 * x_b [B]: the drafted token there.  q = softmax(z / T); T == 0 makes q
 * the point mass on the argmax.  k is capped at V.
 * Outputs: out_k [B] (-1 for an unusable row, SD_DEV_NONFINITE, or an x_b
 *   outside [0, V), SD_DEV_BAD_TOKEN); out_tokens [B, k_max]: the k tokens
 *   of largest logit (ties to the lower id; -0 equals +0), then -1.
 * 1 <= k_max <= 64.  One read of each row.
 * ------------------------------------------------------------------- */
size_t sd_branch_fork_workspace(int B, int V, int k_max, sd_dtype dt);

sd_status sd_branch_fork(const void *draft_logits, sd_dtype dt,
                         const int32_t *x_b, int B, int V, float T, int k_max,
                         int32_t *out_k, int32_t *out_tokens,
                         int32_t *dev_status, void *workspace,
                         size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------
 * Geometric fan-out schedule (Saguaro, Theorem 12).  Host only.
 * F (host) [K+1]: F_0 w_k made integer by largest remainder (ties to the
 * lower k); sum F == budget.  Requires 0 <= K <= SD_MAX_K, budget >= 0,
 * 0 < a < 1, r > 0.
 * ------------------------------------------------------------------- */
sd_status sd_fanout_schedule(int K, int budget, double a, double r,
                             int32_t *F);

/* ---------------------------------------------------------------------
 * Top-F_k per lookahead position (Saguaro, "speculation cache strategy").
 *
 * draft_logits [B, K+1, V]; F (host) [K+1], each F_k in [0, min(V,
 * SD_MAX_FANOUT)].
 * out_tokens [B, sum F] int32: for each k, the F_k token ids with the
 *   largest logit of row k, ordered by (logit descending, id ascending; -0
 *   equals +0), at offset sum_{k' < k} F_{k'}.
 * out_logit [B, sum F] (nullable): their logits.
 * A row holding a NaN gives -1 tokens and SD_DEV_NONFINITE.
 * ------------------------------------------------------------------- */
size_t sd_fanout_topk_workspace(int B, int K, int V, sd_dtype dt);

sd_status sd_fanout_topk(const void *draft_logits, sd_dtype dt, int B, int K,
                         int V, const int32_t *F, int32_t *out_tokens,
                         float *out_logit, int32_t *dev_status,
                         void *workspace, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------
 * Cache hit of the verification outcome (Speculative Speculative Decoding
 * / Saguaro, "technical architecture": the speculator serves the next
 * round from its speculation cache when the verification outcome is in
 * it; "speculation cache strategy": an outcome is (k, t*), k accepted
 * drafts then the correction or bonus token t*, and the cache holds the
 * top-F_k draft tokens of each lookahead position k).
 *
 * n_accepted [B] and out_tokens [B, K+1] as returned by the verify (so
 * t* = out_tokens[b, n_b]); fan_tokens [B, sum F] as returned by
 * sd_fanout_topk with the same F (host [K+1]).  hit [B] int32: 1 if t* is
 * one of the F_{n_b} tokens stored for position n_b, 0 if not, -1 where
 * n_b is outside [0, K] (an unusable row).  All device pointers.
 * ------------------------------------------------------------------- */
sd_status sd_fanout_hits(const int32_t *n_accepted, const int32_t *out_tokens,
                         const int32_t *fan_tokens, int B, int K,
                         const int32_t *F, int32_t *hit, void *stream);

/* ---------------------------------------------------------------------
 * Linear verify fused with the fan-out of the same draft logits, in one
 * launch (the two calls above, same results): the scans of
 * sd_verify_linear, and every CTA left without a sequence to verify (and
 * every resident cluster beyond the B sequences) computes whole fan-out
 * rows, so the fan-out fills the GPU while the last scans finish.  Rows
 * that are not 16-byte aligned (or SD_TUNE_FUSED 0) take the two calls one
 * after the other.
 *
 * draft_logits [B, K+1, V] with K == gamma: rows 0..gamma-1 are the draft
 * rows of the verify, all K+1 rows feed the fan-out.  Other arguments as in
 * sd_verify_linear and sd_fanout_topk (T == 0 is greedy, as there).
 * ------------------------------------------------------------------- */
size_t sd_verify_linear_fanout_workspace(int B, int gamma, int V,
                                         sd_dtype dt);

sd_status sd_verify_linear_fanout(
    const void *target_logits, const void *draft_logits, sd_dtype dt,
    const int32_t *draft_tokens, const float *uniforms, int B, int gamma,
    int V, float T, const int32_t *F, int32_t *n_accepted,
    int32_t *out_tokens, float *out_prob, int32_t *fan_tokens,
    float *fan_logit, int32_t *dev_status, void *workspace, size_t ws_bytes,
    void *stream);

/* ---------------------------------------------------------------------
 * Self-test of the failure path (no counterpart in the pages).  Every
 * wait of a kernel on an asynchronous copy is bounded: after its poll
 * limit it ORs SD_DEV_TIMEOUT into *dev_status and the kernel returns
 * normally.  This call launches one CTA of 256 threads that waits, through
 * that same wait, on a barrier nothing will ever complete (no copy is in
 * flight), with a limit of `polls` in [1, 2^20] polls.
 *
 * dev_status (device, nullable): gets SD_DEV_TIMEOUT.
 * out [2] (device int32): out[0] the number of threads whose wait gave up
 *     (256), out[1] = 1 once the kernel has run to its end.
 * Returns SD_ERR_INVALID_ARG for polls outside the range or a null `out`.
 * ------------------------------------------------------------------- */
sd_status sd_selftest_bounded_wait(int polls, int32_t *dev_status,
                                   int32_t *out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SD_VERIFY_H */
