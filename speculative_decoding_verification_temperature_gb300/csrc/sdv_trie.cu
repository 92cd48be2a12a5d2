// sdv_trie.cu -- K candidate drafts verified as one token tree.
//
// SpecDiff-2 ("core method") samples K candidate drafts independently from
// shared position-wise marginals q_0..q_{gamma-1}; PRESTO (section 2.1)
// verifies a token tree prefix-wise from the root.  Putting the candidates
// in one tree and walking it with the sibling rule of sdv_tree.cu keeps the
// output distributed as the target: the children of a node are the
// candidates' iid draws at that position among the candidates sharing the
// node's prefix.  For that the rule must see every draw, so a token that
// repeats an earlier candidate's token under the same prefix is a leaf
// duplicate (after the first copy is rejected its residual probability is
// 0, so it only applies its residual update) and the candidate continues
// below the first copy.
//
// Layout.  Candidate k's token at position j is node 1 + j K + k (so a
// node's children come in increasing k and increasing node index), node 0
// is the root.  A node that is not a duplicate reads the target row
// (k, j + 1) of the candidate that created it and the draft row j + 1; the
// root reads target row (0, 0) and draft row 0.  Node (k, j) tests with
// uniforms[b][k][j]; the final draw uses uniforms[b][0][gamma].
//
// Two launches: one warp per sequence builds the tree (lane k is candidate
// k; the first earlier lane with the same parent and token is found by
// shuffles), then the tree walk runs with row maps instead of dense node
// rows, so no logit row is copied.
#include "sdv_device.cuh"
#include "sdv_host.cuh"

namespace sdv {

struct TrieOut {
  int32_t *parent, *node_tokens, *trow, *drow, *cand;
  float *uni;
};

__global__ void __launch_bounds__(128)
    trie_build_kernel(const int32_t *tokens, const float *uniforms, int B,
                      int K, int gamma, TrieOut o) {
  const int lane = threadIdx.x & 31;
  const int b = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  if (b >= B) return;  // warp-uniform
  const int N = 1 + K * gamma, G1 = gamma + 1;
  const size_t base = (size_t)b * N;
  const int32_t *x = tokens + (size_t)b * K * gamma;
  const float *u = uniforms + (size_t)b * K * G1;
  const bool live = lane < K;
  if (lane == 0) {
    o.parent[base] = -1;
    o.node_tokens[base] = -1;
    o.uni[base] = u[gamma];
    o.trow[base] = 0;
    o.drow[base] = gamma > 0 ? 0 : -1;
    o.cand[base] = 0;
  }
  int at = 0;  // the node of this candidate's prefix
  for (int j = 0; j < gamma; ++j) {
    const int t = live ? x[(size_t)lane * gamma + j] : 0;
    const int v = 1 + j * K + lane;
    // the first lane with the same prefix node and token
    int first = lane;
    for (int k = 0; k < K; ++k) {
      const int ak = __shfl_sync(0xffffffffu, at, k);
      const int tk = __shfl_sync(0xffffffffu, t, k);
      if (k < first && ak == at && tk == t) first = k;
    }
    const bool dup = first != lane;
    const int own = 1 + j * K + first;  // the first copy (not a duplicate)
    if (live) {
      const size_t i = base + v;
      o.parent[i] = at;
      o.node_tokens[i] = t;
      o.uni[i] = u[(size_t)lane * G1 + j];
      o.cand[i] = lane;
      o.trow[i] = first * G1 + j + 1;
      o.drow[i] = j + 1 < gamma ? j + 1 : -1;
    }
    at = dup ? own : v;
  }
}

}  // namespace sdv

namespace {
size_t align256(size_t x) { return (x + 255) / 256 * 256; }
}  // namespace

extern "C" size_t sd_verify_kcand_trie_workspace(int B, int K, int gamma,
                                                 int V, sd_dtype dt) {
  (void)V;
  (void)dt;
  if (B < 0 || K < 1 || gamma < 0) return 256;
  const size_t n = (size_t)B * (1 + (size_t)K * gamma);
  return 256 + 6 * align256(n * 4);
}

extern "C" sd_status sd_verify_kcand_trie(
    const void *target_logits, const void *draft_logits, sd_dtype dt,
    const int32_t *draft_tokens, const float *uniforms, int B, int K,
    int gamma, int V, float T, int32_t *n_accepted, int32_t *selected_k,
    int32_t *out_tokens, float *out_prob, int32_t *dev_status,
    void *workspace, size_t ws_bytes, void *stream) {
  using namespace sdv;
  SDV_REQUIRE(dt == SD_F32 || dt == SD_BF16, "bad dtype %d", (int)dt);
  SDV_REQUIRE(B >= 0, "B < 0");
  SDV_REQUIRE(K >= 1 && K <= 32, "K=%d outside [1, 32]", K);
  SDV_REQUIRE(gamma >= 0 && gamma <= SD_MAX_GAMMA, "gamma=%d outside [0, %d]",
              gamma, SD_MAX_GAMMA);
  const int N = 1 + K * gamma;
  if (N > SD_MAX_TREE_NODES)
    return fail(SD_ERR_UNSUPPORTED, "1 + K gamma = %d above %d", N,
                SD_MAX_TREE_NODES);
  SDV_REQUIRE(V >= 1 && V <= SD_MAX_V, "V=%d outside [1, %d]", V, SD_MAX_V);
  SDV_REQUIRE(T >= 0.f && std::isfinite(T), "T must be finite and >= 0");
  if (B == 0) return SD_OK;
  SDV_REQUIRE(target_logits && (draft_tokens || gamma == 0) && uniforms &&
                  n_accepted && out_tokens,
              "null pointer");
  SDV_REQUIRE(T == 0.f || gamma == 0 || draft_logits,
              "draft_logits are required when T > 0");
  const size_t need = sd_verify_kcand_trie_workspace(B, K, gamma, V, dt);
  if (!workspace || ws_bytes < need)
    return fail(SD_ERR_INVALID_ARG, "workspace of >= %zu bytes required",
                need);
  const size_t arr = align256((size_t)B * N * 4);
  char *w = static_cast<char *>(workspace) + 256;
  TrieOut o;
  o.parent = reinterpret_cast<int32_t *>(w);
  o.node_tokens = reinterpret_cast<int32_t *>(w + arr);
  o.trow = reinterpret_cast<int32_t *>(w + 2 * arr);
  o.drow = reinterpret_cast<int32_t *>(w + 3 * arr);
  o.cand = reinterpret_cast<int32_t *>(w + 4 * arr);
  o.uni = reinterpret_cast<float *>(w + 5 * arr);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int warps_per_block = 4;
  const int blocks = (B + warps_per_block - 1) / warps_per_block;
  trie_build_kernel<<<blocks, 32 * warps_per_block, 0, s>>>(
      draft_tokens, uniforms, B, K, gamma, o);
  SDV_CUDA(cudaGetLastError());
  TreeMaps m;
  m.trow = o.trow;
  m.drow = o.drow;
  m.trows = K * (gamma + 1);
  m.drows = gamma;
  m.out_cols = gamma + 1;
  m.node_cand = o.cand;
  m.out_cand = selected_k;
  // gamma == 0: the root alone, whose last token is drawn from p by either
  // rule; the deterministic-draft walk is the one that reads no draft rows
  return tree_launch(target_logits, T == 0.f ? nullptr : draft_logits, dt,
                     o.parent, o.node_tokens, o.uni, B, N, V, T, gamma == 0,
                     n_accepted, out_tokens, nullptr, out_prob, dev_status,
                     workspace, 256, stream, &m);
}
