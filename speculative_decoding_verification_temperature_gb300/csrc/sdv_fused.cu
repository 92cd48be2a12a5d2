// sdv_fused.cu -- sd_verify_linear_fanout: the linear verify ("01 ·
// Draft-then-verify", Algorithm 1) and the Saguaro fan-out ("speculation
// cache strategy": the top-F_k draft tokens of every lookahead row k) over
// the same draft logits in one launch.
//
// The fused kernel is the linear verify kernel's FAN instantiation
// (sdv_linear.cu): the scans as in sd_verify_linear, and every CTA left
// without a sequence takes fan-out rows, one CTA per row, so the fan-out's
// rows fill the GPU while the last scans finish (and every resident
// cluster beyond the B sequences does fan-out rows from the start).  The
// draft rows 0..n that the scans stream are not read again when their
// records settle them: each scan thread keeps its best vector of the row
// (sdv_fanrow.cuh), from which the row's exact top-F follows unless a
// check fails; only then is the row read whole.  With rows that are not
// 16-byte aligned or SD_TUNE_FUSED 0 the call runs sd_verify_linear and
// sd_fanout_topk one after the other.
#include "sdv_host.cuh"

namespace sdv {

sd_status linear_launch(const void *target, const void *draft, sd_dtype dt,
                        long long d_seq_rows, const int32_t *tokens,
                        const float *uniforms, int B, int gamma, int V,
                        float T, int32_t *n_acc, int32_t *out_tokens,
                        float *out_prob, float *out_accept, float *out_resid,
                        int32_t *dev_status, void *ws, size_t ws_bytes,
                        cudaStream_t stream);
sd_status linear_fan_launch(const void *target, const void *draft,
                            sd_dtype dt, const int32_t *tokens,
                            const float *uniforms, int B, int gamma, int V,
                            float T, const int32_t *F, int32_t *n_acc,
                            int32_t *out_tokens, float *out_prob,
                            int32_t *fan_tokens, float *fan_logit,
                            int32_t *dev_status, void *ws, size_t ws_bytes,
                            cudaStream_t stream);
size_t fan_workspace(int B, int gamma, int V, sd_dtype dt);
bool fan_applicable(const void *target, const void *draft, sd_dtype dt,
                    int V);

}  // namespace sdv

extern "C" size_t sd_verify_linear_fanout_workspace(int B, int gamma, int V,
                                                    sd_dtype dt) {
  const size_t a = sdv::fan_workspace(B, gamma, V, dt);
  const size_t b = sd_verify_linear_workspace(B, gamma, V, dt);
  return a > b ? a : b;
}

extern "C" sd_status sd_verify_linear_fanout(
    const void *target_logits, const void *draft_logits, sd_dtype dt,
    const int32_t *draft_tokens, const float *uniforms, int B, int gamma,
    int V, float T, const int32_t *F, int32_t *n_accepted,
    int32_t *out_tokens, float *out_prob, int32_t *fan_tokens,
    float *fan_logit, int32_t *dev_status, void *workspace, size_t ws_bytes,
    void *stream) {
  using namespace sdv;
  SDV_REQUIRE(dt == SD_F32 || dt == SD_BF16, "bad dtype %d", (int)dt);
  SDV_REQUIRE(B >= 0, "B < 0");
  SDV_REQUIRE(gamma >= 0 && gamma <= SD_MAX_K, "gamma=%d outside [0, %d]",
              gamma, SD_MAX_K);
  SDV_REQUIRE(V >= 1 && V <= SD_MAX_V, "V=%d outside [1, %d]", V, SD_MAX_V);
  SDV_REQUIRE(T >= 0.f && std::isfinite(T), "T must be finite and >= 0");
  SDV_REQUIRE(F != nullptr, "F is null");
  int total = 0;
  for (int k = 0; k <= gamma; ++k) {
    SDV_REQUIRE(F[k] >= 0, "F[%d] < 0", k);
    if (F[k] > SD_MAX_FANOUT || F[k] > V)
      return fail(SD_ERR_UNSUPPORTED, "F[%d]=%d exceeds min(V, %d)", k, F[k],
                  SD_MAX_FANOUT);
    total += F[k];
  }
  if (B == 0) return SD_OK;
  SDV_REQUIRE(target_logits && draft_logits && n_accepted && out_tokens,
              "null pointer");
  SDV_REQUIRE(total == 0 || fan_tokens, "fan_tokens is null");
  SDV_REQUIRE(gamma == 0 || draft_tokens, "draft_tokens is null");
  SDV_REQUIRE(T == 0.f || uniforms, "uniforms is null");
  int sms = 0;
  sd_status st = check_device(&sms);
  if (st != SD_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (tune(SD_TUNE_FUSED) != 0 && total > 0 &&
      fan_applicable(target_logits, draft_logits, dt, V))
    return linear_fan_launch(target_logits, draft_logits, dt, draft_tokens,
                             uniforms, B, gamma, V, T, F, n_accepted,
                             out_tokens, out_prob, fan_tokens, fan_logit,
                             dev_status, workspace, ws_bytes, s);
  // the two calls one after the other (same results)
  st = linear_launch(target_logits, draft_logits, dt, gamma + 1, draft_tokens,
                     uniforms, B, gamma, V, T, n_accepted, out_tokens,
                     out_prob, nullptr, nullptr, dev_status, workspace,
                     ws_bytes, s);
  if (st != SD_OK) return st;
  return sd_fanout_topk(draft_logits, dt, B, gamma, V, F, fan_tokens,
                        fan_logit, dev_status, nullptr, 0, stream);
}
