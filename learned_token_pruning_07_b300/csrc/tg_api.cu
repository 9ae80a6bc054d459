// tg_api.cu — the extern "C" entry points of libtokengate: argument validation on the host,
// then the launches in tg_score.cu / tg_select.cu / tg_gather.cu / tg_attention.cu.
#include <cmath>

#include "tg_common.cuh"

namespace tg_host {
tg_status launch_gate_score(const uint16_t *h, int32_t T, int32_t d, const uint8_t *mask,
                            const uint16_t *W1, const float *b1, const uint16_t *w2, float b2,
                            int32_t d_g, float *s_out, float *g_out, int32_t *status,
                            cudaStream_t stream, bool rmsnorm, float ln_eps, int32_t H_g = 1,
                            const float *b2h = nullptr, float *s_sel = nullptr);
tg_status launch_fold_rmsnorm_weight(const uint16_t *W1, const uint16_t *ln_w, int32_t d_g, int32_t d,
                                     uint16_t *W1_out, cudaStream_t stream);
tg_status launch_topk_select(const float *s, const uint8_t *mask, const int32_t *cu_seqlens,
                             int32_t B, int32_t T, int32_t K, int32_t *kept_idx, int32_t capacity,
                             int32_t *cu_kept, int32_t *status, cudaStream_t stream, int32_t cu_base = 0);
tg_status launch_gather(const uint16_t *h, const int32_t *pos, const float *g, int32_t H_g,
                        const int32_t *cu_seqlens, int32_t B, int32_t T, int32_t d,
                        const int32_t *kept_idx, const int32_t *cu_kept, int32_t capacity,
                        uint16_t *h_kept, int32_t *pos_kept, float *g_kept, int32_t *status,
                        cudaStream_t stream, int32_t B_kept = -1);
tg_status launch_two_budget_prologue(const int32_t *cu_seqlens, int32_t B, int32_t T, int32_t *kept_idx,
                                     int32_t *cu_packed, cudaStream_t stream);
tg_status launch_rope(uint16_t *X, const int32_t *pos, const int32_t *cu_kept, int32_t B,
                      int32_t capacity, int32_t H, int32_t d_h, float theta, cudaStream_t stream);
tg_status launch_gated_attention(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                                 const float *g, int32_t H_g, const int32_t *cu_kept, int32_t B,
                                 int32_t M_cap, int32_t max_seqlen, int32_t H_q, int32_t H_kv,
                                 int32_t d_h, const float *tau, const float *beta, uint16_t *O,
                                 int32_t *status, cudaStream_t stream, float *lse = nullptr,
                                 void *workspace = nullptr, size_t workspace_bytes = 0);
size_t gated_attention_workspace_size(int32_t B, int32_t max_seqlen, int32_t H_q, int32_t H_kv, int32_t d_h);
tg_status launch_gated_attention_noalloc(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                                         const float *g, int32_t H_g, const int32_t *cu_kept, int32_t B,
                                         int32_t M_cap, int32_t max_seqlen, int32_t H_q, int32_t H_kv,
                                         int32_t d_h, const float *tau, const float *beta, uint16_t *O,
                                         int32_t *status, cudaStream_t stream);
tg_status launch_gated_attention_bwd(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                                     const float *g, int32_t H_g, const uint16_t *O, const uint16_t *dO,
                                     const float *lse, const int32_t *cu_kept, int32_t B, int32_t M_cap,
                                     int32_t max_seqlen, int32_t H_q, int32_t H_kv, int32_t d_h,
                                     const float *tau, const float *beta, float *dQ, float *dK, float *dV,
                                     float *dbias, int32_t *status, cudaStream_t stream);
tg_status launch_gate_score_grad(const float *dbias, const float *beta, const float *g_kept, int32_t H_g,
                                 const int32_t *kept_idx, const int32_t *cu_kept, int32_t B,
                                 int32_t capacity, int32_t H_q, int32_t T, float *ds, cudaStream_t stream);
tg_status launch_gated_attention_eq8(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                                     const float *b, int32_t H_g, const int32_t *pos, const int32_t *cu_kept,
                                     int32_t B, int32_t M_cap, int32_t max_seqlen, int32_t H_q,
                                     int32_t H_kv, int32_t d_h, const float *gain,
                                     const float *temp, uint16_t *O, int32_t *status,
                                     cudaStream_t stream);
tg_status launch_normalize_scores(const float *s, int32_t H_g, const uint8_t *mask, const int32_t *cu_seqlens,
                                  int32_t B, int32_t T, float eps, float *b_out, float *b_sel, int32_t *status,
                                  cudaStream_t stream);
}  // namespace tg_host

namespace {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline cudaStream_t S(tg_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

constexpr int32_t kMaxSelectB = 1024;
constexpr int32_t kMaxGateHeads = 16;

// H_g gate heads: 1 <= H_g <= 16, and the query heads split evenly over them
tg_status check_gate_heads(int32_t H_g, int32_t H_q) {
  if (H_g < 1) return TG_ERR_INVALID_ARG;
  if (H_g > kMaxGateHeads || (H_q > 0 && H_q % H_g != 0)) return TG_ERR_UNSUPPORTED;
  return TG_OK;
}

tg_status check_gate_score(const uint16_t *h, int32_t T, int32_t d, const uint16_t *W1,
                           const uint16_t *w2, int32_t d_g, const float *s_out, float b2) {
  if (!h || !W1 || !w2 || !s_out) return TG_ERR_INVALID_ARG;
  if (T < 0 || d <= 0 || d_g <= 0 || !std::isfinite(b2)) return TG_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(W1)) return TG_ERR_INVALID_ARG;
  if (d % 32 != 0 || d_g % 32 != 0 || d_g > 512) return TG_ERR_UNSUPPORTED;
  return TG_OK;
}

tg_status check_select(const float *s, const int32_t *cu_seqlens, int32_t B, int32_t T, int32_t K,
                       const int32_t *kept_idx, int32_t capacity, const int32_t *cu_kept) {
  if (!s || !cu_seqlens || !cu_kept) return TG_ERR_INVALID_ARG;
  if (B < 1 || T < 0 || K < 0 || capacity < 0) return TG_ERR_INVALID_ARG;
  if (capacity > 0 && !kept_idx) return TG_ERR_INVALID_ARG;
  if (B > kMaxSelectB) return TG_ERR_UNSUPPORTED;
  return TG_OK;
}

tg_status check_gather(const uint16_t *h, const int32_t *cu_seqlens, int32_t B, int32_t T,
                       int32_t d, const int32_t *kept_idx, const int32_t *cu_kept,
                       int32_t capacity, const uint16_t *h_kept) {
  if (!h || !cu_seqlens || !kept_idx || !cu_kept || !h_kept) return TG_ERR_INVALID_ARG;
  if (B < 1 || T < 0 || d <= 0 || capacity < 0) return TG_ERR_INVALID_ARG;
  if (d % 8 != 0 || !aligned16(h) || !aligned16(h_kept)) return TG_ERR_INVALID_ARG;
  return TG_OK;
}

}  // namespace

extern "C" {

tg_status tg_gate_score(const uint16_t *h, int32_t T_total, int32_t d, const uint8_t *instr_mask,
                        const uint16_t *W1, const float *b1, const uint16_t *w2, float b2,
                        int32_t d_g, float *s_out, float *g_out, int32_t *status,
                        tg_stream_t stream) {
  tg_status st = check_gate_score(h, T_total, d, W1, w2, d_g, s_out, b2);
  if (st != TG_OK) return st;
  return tg_host::launch_gate_score(h, T_total, d, instr_mask, W1, b1, w2, b2, d_g, s_out, g_out,
                                    status, S(stream), false, 0.0f);
}

tg_status tg_gate_score_rmsnorm(const uint16_t *h, int32_t T_total, int32_t d,
                                const uint8_t *instr_mask, const uint16_t *W1_folded, const float *b1,
                                const uint16_t *w2, float b2, int32_t d_g, float ln_eps, float *s_out,
                                float *g_out, int32_t *status, tg_stream_t stream) {
  tg_status st = check_gate_score(h, T_total, d, W1_folded, w2, d_g, s_out, b2);
  if (st != TG_OK) return st;
  if (!std::isfinite(ln_eps) || ln_eps < 0.0f) return TG_ERR_INVALID_ARG;
  return tg_host::launch_gate_score(h, T_total, d, instr_mask, W1_folded, b1, w2, b2, d_g, s_out, g_out,
                                    status, S(stream), true, ln_eps);
}

tg_status tg_gate_score_heads(const uint16_t *h, int32_t T_total, int32_t d, const uint8_t *instr_mask,
                              const uint16_t *W1, const float *b1, const uint16_t *W2, const float *b2,
                              int32_t d_g, int32_t H_g, int32_t rmsnorm, float ln_eps, float *s_heads,
                              float *g_heads, float *s_sel, int32_t *status, tg_stream_t stream) {
  tg_status st = check_gate_score(h, T_total, d, W1, W2, d_g, s_heads, 0.0f);
  if (st == TG_OK) st = check_gate_heads(H_g, 0);
  if (st != TG_OK) return st;
  if (!s_sel || (rmsnorm != 0 && rmsnorm != 1)) return TG_ERR_INVALID_ARG;
  if (rmsnorm && (!std::isfinite(ln_eps) || ln_eps < 0.0f)) return TG_ERR_INVALID_ARG;
  for (int c = 0; b2 && c < H_g; ++c)
    if (!std::isfinite(b2[c])) return TG_ERR_INVALID_ARG;
  return tg_host::launch_gate_score(h, T_total, d, instr_mask, W1, b1, W2, b2 ? b2[0] : 0.0f, d_g, s_heads,
                                    g_heads, status, S(stream), rmsnorm != 0, ln_eps, H_g, b2, s_sel);
}

tg_status tg_fold_rmsnorm_weight(const uint16_t *W1, const uint16_t *ln_weight, int32_t d_g, int32_t d,
                                 uint16_t *W1_out, tg_stream_t stream) {
  if (!W1 || !ln_weight || !W1_out || d_g <= 0 || d <= 0) return TG_ERR_INVALID_ARG;
  return tg_host::launch_fold_rmsnorm_weight(W1, ln_weight, d_g, d, W1_out, S(stream));
}

tg_status tg_topk_select(const float *s, const uint8_t *instr_mask, const int32_t *cu_seqlens,
                         int32_t B, int32_t T_total, int32_t K, int32_t *kept_idx,
                         int32_t capacity, int32_t *cu_kept, int32_t *status, tg_stream_t stream) {
  tg_status st = check_select(s, cu_seqlens, B, T_total, K, kept_idx, capacity, cu_kept);
  if (st != TG_OK) return st;
  return tg_host::launch_topk_select(s, instr_mask, cu_seqlens, B, T_total, K, kept_idx, capacity,
                                     cu_kept, status, S(stream));
}

tg_status tg_gather_kept(const uint16_t *h, const int32_t *pos, const float *g, int32_t H_g,
                         const int32_t *cu_seqlens, int32_t B, int32_t T_total, int32_t d,
                         const int32_t *kept_idx, const int32_t *cu_kept, int32_t capacity,
                         uint16_t *h_kept, int32_t *pos_kept, float *g_kept, int32_t *status,
                         tg_stream_t stream) {
  tg_status st = check_gather(h, cu_seqlens, B, T_total, d, kept_idx, cu_kept, capacity, h_kept);
  if (st == TG_OK) st = check_gate_heads(H_g, 0);
  if (st != TG_OK) return st;
  return tg_host::launch_gather(h, pos, g, H_g, cu_seqlens, B, T_total, d, kept_idx, cu_kept, capacity,
                                h_kept, pos_kept, g_kept, status, S(stream));
}

namespace {
tg_status check_attention(const uint16_t *Q, const uint16_t *K, const uint16_t *V, int32_t H_g,
                          const int32_t *cu_kept, int32_t B, int32_t M_capacity, int32_t max_seqlen,
                          int32_t H_q, int32_t H_kv, int32_t d_h, const float *tau, const float *beta,
                          const void *O) {
  if (!Q || !K || !V || !cu_kept || !tau || !beta || !O || H_g < 1) return TG_ERR_INVALID_ARG;
  if (B < 1 || M_capacity < 0 || max_seqlen < 0 || H_q < 1 || H_kv < 1 || d_h < 1)
    return TG_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return TG_ERR_INVALID_ARG;
  for (int h = 0; h < H_q && h < 128; ++h) {
    if (!std::isfinite(tau[h]) || !(tau[h] > 0.0f)) return TG_ERR_INVALID_ARG;
    if (!std::isfinite(beta[h]) || beta[h] < 0.0f) return TG_ERR_INVALID_ARG;
  }
  if (H_q % H_kv != 0 || H_q > 128 || (d_h != 128 && d_h != 64)) return TG_ERR_UNSUPPORTED;
  return check_gate_heads(H_g, H_q);
}
}  // namespace

tg_status tg_gated_attention(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                             const float *g, int32_t H_g, const int32_t *cu_kept, int32_t B,
                             int32_t M_capacity, int32_t max_seqlen, int32_t H_q, int32_t H_kv,
                             int32_t d_h, const float *tau, const float *beta, uint16_t *O,
                             int32_t *status, tg_stream_t stream) {
  tg_status st = check_attention(Q, K, V, H_g, cu_kept, B, M_capacity, max_seqlen, H_q, H_kv, d_h, tau, beta, O);
  if (st != TG_OK) return st;
  return tg_host::launch_gated_attention(Q, K, V, g, H_g, cu_kept, B, M_capacity, max_seqlen, H_q, H_kv,
                                         d_h, tau, beta, O, status, S(stream));
}

size_t tg_gated_attention_workspace_size(int32_t B, int32_t max_seqlen, int32_t H_q, int32_t H_kv, int32_t d_h) {
  return tg_host::gated_attention_workspace_size(B, max_seqlen, H_q, H_kv, d_h);
}

tg_status tg_gated_attention_ws(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                                const float *g, int32_t H_g, const int32_t *cu_kept, int32_t B,
                                int32_t M_capacity, int32_t max_seqlen, int32_t H_q, int32_t H_kv,
                                int32_t d_h, const float *tau, const float *beta, uint16_t *O,
                                void *workspace, size_t workspace_bytes, int32_t *status,
                                tg_stream_t stream) {
  tg_status st = check_attention(Q, K, V, H_g, cu_kept, B, M_capacity, max_seqlen, H_q, H_kv, d_h, tau, beta, O);
  if (st != TG_OK) return st;
  if (workspace == nullptr && workspace_bytes != 0) return TG_ERR_INVALID_ARG;
  return tg_host::launch_gated_attention(Q, K, V, g, H_g, cu_kept, B, M_capacity, max_seqlen, H_q, H_kv,
                                         d_h, tau, beta, O, status, S(stream), nullptr, workspace,
                                         workspace_bytes);
}

tg_status tg_gated_attention_noalloc(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                                     const float *g, int32_t H_g, const int32_t *cu_kept, int32_t B,
                                     int32_t M_capacity, int32_t max_seqlen, int32_t H_q, int32_t H_kv,
                                     int32_t d_h, const float *tau, const float *beta, uint16_t *O,
                                     int32_t *status, tg_stream_t stream) {
  const tg_status st =
      check_attention(Q, K, V, H_g, cu_kept, B, M_capacity, max_seqlen, H_q, H_kv, d_h, tau, beta, O);
  if (st != TG_OK) return st;
  return tg_host::launch_gated_attention_noalloc(Q, K, V, g, H_g, cu_kept, B, M_capacity, max_seqlen, H_q,
                                                 H_kv, d_h, tau, beta, O, status, S(stream));
}

tg_status tg_gated_attention_lse(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                                 const float *g, int32_t H_g, const int32_t *cu_kept, int32_t B,
                                 int32_t M_capacity, int32_t max_seqlen, int32_t H_q, int32_t H_kv,
                                 int32_t d_h, const float *tau, const float *beta, uint16_t *O,
                                 float *lse, int32_t *status, tg_stream_t stream) {
  tg_status st = check_attention(Q, K, V, H_g, cu_kept, B, M_capacity, max_seqlen, H_q, H_kv, d_h, tau, beta, O);
  if (st == TG_OK && !lse) st = TG_ERR_INVALID_ARG;
  if (st != TG_OK) return st;
  return tg_host::launch_gated_attention(Q, K, V, g, H_g, cu_kept, B, M_capacity, max_seqlen, H_q, H_kv,
                                         d_h, tau, beta, O, status, S(stream), lse);
}

tg_status tg_gated_attention_bwd(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                                 const float *g, int32_t H_g, const uint16_t *O, const uint16_t *dO,
                                 const float *lse, const int32_t *cu_kept, int32_t B,
                                 int32_t M_capacity, int32_t max_seqlen, int32_t H_q, int32_t H_kv,
                                 int32_t d_h, const float *tau, const float *beta, float *dQ,
                                 float *dK, float *dV, float *dbias, int32_t *status,
                                 tg_stream_t stream) {
  tg_status st = check_attention(Q, K, V, H_g, cu_kept, B, M_capacity, max_seqlen, H_q, H_kv, d_h, tau, beta, O);
  if (st == TG_OK && (!dO || !lse || !dQ || !dK || !dV || !dbias)) st = TG_ERR_INVALID_ARG;
  if (st != TG_OK) return st;
  return tg_host::launch_gated_attention_bwd(Q, K, V, g, H_g, O, dO, lse, cu_kept, B, M_capacity, max_seqlen,
                                             H_q, H_kv, d_h, tau, beta, dQ, dK, dV, dbias, status,
                                             S(stream));
}

tg_status tg_gate_score_grad(const float *dbias, const float *beta, const float *g_kept, int32_t H_g,
                             const int32_t *kept_idx, const int32_t *cu_kept, int32_t B,
                             int32_t capacity, int32_t H_q, int32_t T_total, float *ds,
                             tg_stream_t stream) {
  if (!dbias || !beta || !g_kept || !kept_idx || !cu_kept || !ds) return TG_ERR_INVALID_ARG;
  if (B < 1 || capacity < 0 || H_q < 1 || H_q > 128 || T_total < 0) return TG_ERR_INVALID_ARG;
  for (int h = 0; h < H_q; ++h)
    if (!std::isfinite(beta[h])) return TG_ERR_INVALID_ARG;
  const tg_status st = check_gate_heads(H_g, H_q);
  if (st != TG_OK) return st;
  return tg_host::launch_gate_score_grad(dbias, beta, g_kept, H_g, kept_idx, cu_kept, B, capacity, H_q, T_total, ds,
                                         S(stream));
}

tg_status tg_normalize_scores(const float *s, int32_t H_g, const uint8_t *instr_mask, const int32_t *cu_seqlens,
                              int32_t B, int32_t T_total, float eps, float *b_out, float *b_sel, int32_t *status,
                              tg_stream_t stream) {
  if (!s || !cu_seqlens || !b_out) return TG_ERR_INVALID_ARG;
  if (B < 1 || T_total < 0 || !std::isfinite(eps) || eps < 0.0f) return TG_ERR_INVALID_ARG;
  const tg_status st = check_gate_heads(H_g, 0);
  if (st != TG_OK) return st;
  if (B > kMaxSelectB) return TG_ERR_UNSUPPORTED;
  if (T_total == 0) return TG_OK;
  return tg_host::launch_normalize_scores(s, H_g, instr_mask, cu_seqlens, B, T_total, eps, b_out, b_sel, status,
                                          S(stream));
}

tg_status tg_gated_attention_eq8(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                                 const float *b, int32_t H_g, const int32_t *pos, const int32_t *cu_kept,
                                 int32_t B, int32_t M_capacity, int32_t max_seqlen, int32_t H_q,
                                 int32_t H_kv, int32_t d_h, const float *gain, const float *temp,
                                 uint16_t *O, int32_t *status, tg_stream_t stream) {
  if (!Q || !K || !V || !pos || !cu_kept || !gain || !temp || !O) return TG_ERR_INVALID_ARG;
  if (B < 1 || M_capacity < 0 || max_seqlen < 0 || H_q < 1 || H_kv < 1 || d_h < 1)
    return TG_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return TG_ERR_INVALID_ARG;
  for (int h = 0; h < H_q && h < 128; ++h) {
    if (!std::isfinite(gain[h]) || gain[h] < 0.0f) return TG_ERR_INVALID_ARG;
    if (!std::isfinite(temp[h]) || temp[h] < 0.0f) return TG_ERR_INVALID_ARG;
  }
  if (H_q % H_kv != 0 || H_q > 128 || (d_h != 128 && d_h != 64)) return TG_ERR_UNSUPPORTED;
  const tg_status st = check_gate_heads(H_g, H_q);
  if (st != TG_OK) return st;
  return tg_host::launch_gated_attention_eq8(Q, K, V, b, H_g, pos, cu_kept, B, M_capacity, max_seqlen, H_q,
                                             H_kv, d_h, gain, temp, O, status, S(stream));
}

tg_status tg_gate_prune_layer(const uint16_t *h, const int32_t *pos, const uint8_t *instr_mask,
                              const int32_t *cu_seqlens, int32_t B, int32_t T_total, int32_t d,
                              const uint16_t *W1, const float *b1, const uint16_t *w2, float b2,
                              int32_t d_g, int32_t K, float *s_out, float *g_out,
                              int32_t *kept_idx, int32_t capacity, int32_t *cu_kept,
                              uint16_t *h_kept, int32_t *pos_kept, float *g_kept,
                              int32_t *status, tg_stream_t stream) {
  tg_status st = check_gate_score(h, T_total, d, W1, w2, d_g, s_out, b2);
  if (st == TG_OK && !g_out) st = TG_ERR_INVALID_ARG;
  if (st == TG_OK) st = check_select(s_out, cu_seqlens, B, T_total, K, kept_idx, capacity, cu_kept);
  if (st == TG_OK)
    st = check_gather(h, cu_seqlens, B, T_total, d, kept_idx, cu_kept, capacity, h_kept);
  if (st != TG_OK) return st;
  st = tg_host::launch_gate_score(h, T_total, d, instr_mask, W1, b1, w2, b2, d_g, s_out, g_out,
                                  status, S(stream), false, 0.0f);
  if (st != TG_OK) return st;
  st = tg_host::launch_topk_select(s_out, instr_mask, cu_seqlens, B, T_total, K, kept_idx,
                                   capacity, cu_kept, status, S(stream));
  if (st != TG_OK) return st;
  return tg_host::launch_gather(h, pos, g_out, 1, cu_seqlens, B, T_total, d, kept_idx, cu_kept,
                                capacity, h_kept, pos_kept, g_kept, status, S(stream));
}

tg_status tg_gate_prune_layer_heads(const uint16_t *h, const int32_t *pos, const uint8_t *instr_mask,
                                    const int32_t *cu_seqlens, int32_t B, int32_t T_total, int32_t d,
                                    const uint16_t *W1, const float *b1, const uint16_t *W2, const float *b2,
                                    int32_t d_g, int32_t H_g, int32_t K, float *s_heads, float *g_heads,
                                    float *s_sel, int32_t *kept_idx, int32_t capacity, int32_t *cu_kept,
                                    uint16_t *h_kept, int32_t *pos_kept, float *g_kept, int32_t *status,
                                    tg_stream_t stream) {
  tg_status st = check_gate_score(h, T_total, d, W1, W2, d_g, s_heads, 0.0f);
  if (st == TG_OK) st = check_gate_heads(H_g, 0);
  if (st == TG_OK && (!g_heads || !s_sel)) st = TG_ERR_INVALID_ARG;
  if (st == TG_OK) st = check_select(s_sel, cu_seqlens, B, T_total, K, kept_idx, capacity, cu_kept);
  if (st == TG_OK)
    st = check_gather(h, cu_seqlens, B, T_total, d, kept_idx, cu_kept, capacity, h_kept);
  for (int c = 0; st == TG_OK && b2 && c < H_g; ++c)
    if (!std::isfinite(b2[c])) st = TG_ERR_INVALID_ARG;
  if (st != TG_OK) return st;
  st = tg_host::launch_gate_score(h, T_total, d, instr_mask, W1, b1, W2, b2 ? b2[0] : 0.0f, d_g, s_heads,
                                  g_heads, status, S(stream), false, 0.0f, H_g, b2, s_sel);
  if (st != TG_OK) return st;
  st = tg_host::launch_topk_select(s_sel, instr_mask, cu_seqlens, B, T_total, K, kept_idx, capacity, cu_kept,
                                   status, S(stream));
  if (st != TG_OK) return st;
  return tg_host::launch_gather(h, pos, g_heads, H_g, cu_seqlens, B, T_total, d, kept_idx, cu_kept, capacity,
                                h_kept, pos_kept, g_kept, status, S(stream));
}

tg_status tg_two_budget_prune_layer(const uint16_t *h, const int32_t *pos, const uint8_t *instr_mask,
                                    const int32_t *cu_seqlens, int32_t B, int32_t T_total, int32_t d,
                                    const uint16_t *W1, const float *b1, const uint16_t *w2, float b2,
                                    int32_t d_g, int32_t K_prune, float *s_out, float *g_out,
                                    int32_t *kept_idx, int32_t capacity, int32_t *cu_packed,
                                    uint16_t *h_kept, int32_t *pos_kept, float *g_kept,
                                    int32_t *status, tg_stream_t stream) {
  tg_status st = check_gate_score(h, T_total, d, W1, w2, d_g, s_out, b2);
  if (st == TG_OK && !g_out) st = TG_ERR_INVALID_ARG;
  if (st == TG_OK && capacity < T_total) st = TG_ERR_INVALID_ARG;  // the full half alone is T_total rows
  if (st == TG_OK) st = check_select(s_out, cu_seqlens, B, T_total, K_prune, kept_idx, capacity, cu_packed);
  if (st == TG_OK)
    st = check_gather(h, cu_seqlens, B, T_total, d, kept_idx, cu_packed, capacity, h_kept);
  if (st == TG_OK && B > kMaxSelectB / 2) st = TG_ERR_UNSUPPORTED;
  if (st != TG_OK) return st;
  st = tg_host::launch_gate_score(h, T_total, d, instr_mask, W1, b1, w2, b2, d_g, s_out, g_out,
                                  status, S(stream), false, 0.0f);
  if (st != TG_OK) return st;
  st = tg_host::launch_two_budget_prologue(cu_seqlens, B, T_total, kept_idx, cu_packed, S(stream));
  if (st != TG_OK) return st;
  st = tg_host::launch_topk_select(s_out, instr_mask, cu_seqlens, B, T_total, K_prune, kept_idx + T_total,
                                   capacity - T_total, cu_packed + B, status, S(stream), T_total);
  if (st != TG_OK) return st;
  return tg_host::launch_gather(h, pos, g_out, 1, cu_seqlens, B, T_total, d, kept_idx, cu_packed, capacity,
                                h_kept, pos_kept, g_kept, status, S(stream), 2 * B);
}

tg_status tg_apply_rope(uint16_t *X, const int32_t *pos, const int32_t *cu_kept, int32_t B,
                        int32_t capacity, int32_t H, int32_t d_h, float theta,
                        tg_stream_t stream) {
  if (!X || !pos) return TG_ERR_INVALID_ARG;
  if (capacity < 0 || H < 1 || d_h < 2 || d_h % 2 != 0 || !(theta > 0.0f) || !std::isfinite(theta))
    return TG_ERR_INVALID_ARG;
  if (cu_kept && B < 1) return TG_ERR_INVALID_ARG;
  if (d_h > 256) return TG_ERR_UNSUPPORTED;
  return tg_host::launch_rope(X, pos, cu_kept, B, capacity, H, d_h, theta, S(stream));
}

}  // extern "C"
