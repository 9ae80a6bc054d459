/*
 * tokengate.h — C ABI of libtokengate, the B300 (sm_103a) TokenGate gated-prefill path.
 *
 * The path (TokenGate paper deep dive, agientry.com, sections 3.1-3.4; TokenGate paper
 * page, thelatestinai.com, Figure 1): at the gate layer a small MLP scores every hidden
 * state, a top-K selector keeps the K highest-scoring document tokens plus every
 * non-prunable (instruction / question) token in original order, the kept rows, their
 * original position ids and gate values are gathered, and the layers above run
 * token-gated causal GQA attention over the kept tokens only.
 *
 * Conventions shared by every entry point
 *  - Every function returns a tg_status. TG_OK means the work was enqueued (or done).
 *  - Pointers marked [device] are device memory owned by the caller; the library never
 *    allocates, frees or retains them beyond the call. Pointers marked [host] are read
 *    during the call only.
 *  - bf16 tensors are passed as uint16_t* holding bf16 bit patterns.
 *  - All work is enqueued asynchronously on the caller's stream (NULL = legacy default).
 *  - Host scalars are validated before anything is launched; a bad one returns
 *    TG_ERR_INVALID_ARG (or TG_ERR_UNSUPPORTED for a legal shape the kernels do not
 *    tile) and launches nothing.
 *  - Conditions only the device can see (cu_seqlens that are not a non-decreasing
 *    partition of [0, T_total], an index out of range, an output that would pass its
 *    capacity, a pipeline wait that gave up) are reported through the caller's int32
 *    `status` word in device memory: the kernels OR in a TG_DEV_* bit and never touch
 *    memory out of bounds. The caller zeroes the word; tg_read_device_status() fetches it.
 *  - Launch errors are returned as TG_ERR_CUDA; tg_last_cuda_error() gives the code.
 *  - No NaN policy is imposed on data; top-K ranks NaN below every number.
 */
#ifndef TOKENGATE_H_
#define TOKENGATE_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TG_API __attribute__((visibility("default")))
#else
#define TG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *tg_stream_t; /* the same handle as cudaStream_t */

typedef int32_t tg_status;
enum {
  TG_OK = 0,
  TG_ERR_INVALID_ARG = 1,
  TG_ERR_UNSUPPORTED = 2,
  TG_ERR_CUDA = 3,
  TG_ERR_CAPACITY = 4,
  TG_ERR_DEVICE_TIMEOUT = 5,
  TG_ERR_DEVICE = 6
};

/* Bits the kernels OR into the caller's device status word. */
enum {
  TG_DEV_BAD_SEQLENS = 1 << 0, /* cu_seqlens / cu_kept not a valid partition          */
  TG_DEV_BAD_INDEX = 1 << 1,   /* a kept index outside [0, T_total)                      */
  TG_DEV_CAPACITY = 1 << 2,    /* output would pass its capacity; the excess was dropped */
  TG_DEV_TIMEOUT = 1 << 3      /* a pipeline wait gave up; outputs are not valid          */
};

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
TG_API int32_t tg_version(void);

/* Human-readable name of a status code (static storage). */
TG_API const char *tg_status_string(tg_status s);

/* The last CUDA runtime error seen by any entry point on this thread (cudaError_t value). */
TG_API int32_t tg_last_cuda_error(void);

/*
 * tg_gate_score — score every row (deep dive section 3.1, Eq. (3): b~_j = MLP(a~_j)).
 *   u = W1 h_j (+ b1), s_j = w2 . SiLU(u) (+ b2), g_j = sigmoid(s_j); g_j = 1 on
 *   non-prunable rows (they carry zero log-bias, the reading of "b_j := 0 for j in N").
 *   h          [device] bf16 [T_total, d], row-major (token-major), 16-byte aligned.
 *   instr_mask [device] uint8 [T_total], 1 = non-prunable. May be NULL (no such rows).
 *   W1         [device] bf16 [d_g, d], row-major, 16-byte aligned.
 *   b1         [device] fp32 [d_g] or NULL.   w2 [device] bf16 [d_g].   b2: host scalar.
 *   s_out      [device] fp32 [T_total]: the fp32 score that top-K ranks.
 *   g_out      [device] fp32 [T_total]: the gate value. May be NULL.
 *   status     [device] int32 word (TG_DEV_TIMEOUT).
 *   Shapes: d % 32 == 0, d_g % 32 == 0, 32 <= d_g <= 512; else TG_ERR_UNSUPPORTED.
 *   Compute: bf16 tcgen05 MMA with fp32 accumulation in tensor memory; fp32 epilogue.
 */
TG_API tg_status tg_gate_score(const uint16_t *h, int32_t T_total, int32_t d, const uint8_t *instr_mask,
                        const uint16_t *W1, const float *b1, const uint16_t *w2, float b2,
                        int32_t d_g, float *s_out, float *g_out, int32_t *status,
                        tg_stream_t stream);

/*
 * tg_gate_score_rmsnorm — tg_gate_score with LN_2 fused in front of the score MLP (deep dive
 *   section 2, Eq. (1): the gate scores the normalised post-attention residual
 *   a~ = LN_2(a^L); in the Qwen3 family LN_2 is an RMSNorm with a weight w_ln):
 *     u = W1 (w_ln * h / sqrt(mean_c h_c^2 + ln_eps)) (+ b1), then as tg_gate_score.
 *   h is the raw residual a^L. W1_folded [device] bf16 [d_g, d] = W1 diag(w_ln) rounded to
 *   bf16, as written by tg_fold_rmsnorm_weight; the kernel sums each row's squares while the
 *   row streams through shared memory and scales the row's accumulator by 1/rms, so the
 *   normalised activations never go to memory. ln_eps: host, finite, >= 0.
 *   Other arguments, shapes and errors as tg_gate_score.
 */
TG_API tg_status tg_gate_score_rmsnorm(const uint16_t *h, int32_t T_total, int32_t d,
                                const uint8_t *instr_mask, const uint16_t *W1_folded, const float *b1,
                                const uint16_t *w2, float b2, int32_t d_g, float ln_eps, float *s_out,
                                float *g_out, int32_t *status, tg_stream_t stream);

/*
 * tg_gate_score_heads — per-head gate scores (deep dive section 3.4: the gate carries a
 *   per-head bias, and selection aggregates the heads uniformly):
 *     u = W1 a_j (+ b1), s_jc = W2[c] . SiLU(u) (+ b2[c]), g_jc = sigmoid(s_jc) (1 on
 *     non-prunable rows), s_sel_j = (1/H_g) sum_c s_jc (summed in head order in fp32).
 *   W2 [device] bf16 [H_g, d_g], row c the second layer of gate head c; b2 [host] fp32 [H_g]
 *   or NULL. 1 <= H_g <= 16 (else TG_ERR_UNSUPPORTED).
 *   rmsnorm: 0, or 1 for LN_2 fused in front (then W1 is the folded weight and h the raw
 *   residual, as tg_gate_score_rmsnorm; ln_eps finite, >= 0).
 *   s_heads [device] fp32 [T_total, H_g]; g_heads [device] fp32 [T_total, H_g] or NULL;
 *   s_sel [device] fp32 [T_total] (required): the row mean that tg_topk_select ranks.
 *   Other arguments, shapes and errors as tg_gate_score.
 */
TG_API tg_status tg_gate_score_heads(const uint16_t *h, int32_t T_total, int32_t d, const uint8_t *instr_mask,
                              const uint16_t *W1, const float *b1, const uint16_t *W2, const float *b2,
                              int32_t d_g, int32_t H_g, int32_t rmsnorm, float ln_eps, float *s_heads,
                              float *g_heads, float *s_sel, int32_t *status, tg_stream_t stream);

/*
 * tg_fold_rmsnorm_weight — W1_out[k, c] = bf16(W1[k, c] * ln_weight[c]) (round to nearest
 *   even), the weight tg_gate_score_rmsnorm takes. W1 [device] bf16 [d_g, d]; ln_weight
 *   [device] bf16 [d]; W1_out [device] bf16 [d_g, d] (may not alias W1). Run once per weight.
 */
TG_API tg_status tg_fold_rmsnorm_weight(const uint16_t *W1, const uint16_t *ln_weight, int32_t d_g,
                                 int32_t d, uint16_t *W1_out, tg_stream_t stream);

/*
 * tg_topk_select — the retained set (deep dive section 3.1, Eq. (4): S = topK_{j in P}(b_j)
 *   union N; section 3.4: the budget is clamped to |P| and the keep indices are built over
 *   the full sequence in original order).
 *   For each sequence b: K_b = min(K, |P_b|) document rows with the largest s (ties to the
 *   lower row; -0.0 ranks as +0.0; NaN below every number), plus every row with
 *   instr_mask = 1, written in ascending row order.
 *   s          [device] fp32 [T_total].     instr_mask [device] uint8 [T_total] or NULL.
 *   cu_seqlens [device] int32 [B+1], a non-decreasing partition of [0, T_total].
 *   kept_idx   [device] int32 [capacity]: global row of each kept token.
 *   cu_kept    [device] int32 [B+1]: cu_kept[b+1] - cu_kept[b] = K_b + |N_b|.
 *   A capacity of T_total is always enough. Rows past capacity are dropped and
 *   TG_DEV_CAPACITY is set; cu_kept still reports the untruncated counts.
 *   Limits: 1 <= B <= 1024 (else TG_ERR_UNSUPPORTED), K >= 0.
 */
TG_API tg_status tg_topk_select(const float *s, const uint8_t *instr_mask, const int32_t *cu_seqlens,
                         int32_t B, int32_t T_total, int32_t K, int32_t *kept_idx,
                         int32_t capacity, int32_t *cu_kept, int32_t *status, tg_stream_t stream);

/*
 * tg_gather_kept — slice the hidden states and gather the original position ids and gate
 *   values of the kept rows (deep dive section 3.4: hidden_states[:, keep] and
 *   position_ids[:, keep]; paper page Figure 1 (b): kept states travel with their scores).
 *   h        [device] bf16 [T_total, d], 16-byte aligned rows (d % 8 == 0).
 *   pos      [device] int32 [T_total] or NULL (then pos = row - cu_seqlens[b]).
 *   g        [device] fp32 [T_total, H_g] or NULL (then g_kept is not written); H_g gate
 *            values per row (1 <= H_g <= 16; 1 for the single gate).
 *   kept_idx, cu_kept as written by tg_topk_select; rows m < min(cu_kept[B], capacity).
 *   h_kept   [device] bf16 [capacity, d].  pos_kept [device] int32 [capacity] or NULL.
 *   g_kept   [device] fp32 [capacity, H_g] or NULL.
 *   status   [device] int32 word (TG_DEV_BAD_INDEX) or NULL.
 */
TG_API tg_status tg_gather_kept(const uint16_t *h, const int32_t *pos, const float *g, int32_t H_g,
                         const int32_t *cu_seqlens, int32_t B, int32_t T_total, int32_t d,
                         const int32_t *kept_idx, const int32_t *cu_kept, int32_t capacity,
                         uint16_t *h_kept, int32_t *pos_kept, float *g_kept, int32_t *status,
                         tg_stream_t stream);

/*
 * tg_gated_attention — token-gated causal GQA attention over the kept tokens
 *   (deep dive section 3.2, Eq. (5) and Eq. (8), in log-bias form):
 *     o_i = sum_{j <= i, same sequence} softmax_j(tau_h q_i.k_j / sqrt(d_h) + beta_h ln g_j) v_j
 *   With beta_h = 1 each attention weight is multiplied by its key's gate value and
 *   renormalised (paper page Figure 1 (c)). beta_h ln g_j is taken as 0 when beta_h = 0.
 *   Query head h reads kv head h / (H_q / H_kv). A query whose every key has zero weight
 *   outputs zeros.
 *   Q [device] bf16 [M, H_q, d_h];  K, V [device] bf16 [M, H_kv, d_h]; token-major, dense.
 *   g [device] fp32 [M, H_g] or NULL (no bias). Per-head gates (deep dive section 3.4: a
 *     per-head bias): query head h reads g[j, h / (H_q / H_g)]; H_g = 1 is the shared gate.
 *     1 <= H_g <= 16 and H_q % H_g == 0 (else TG_ERR_UNSUPPORTED); pass 1 when g is NULL.
 *   cu_kept [device] int32 [B+1]: sequence boundaries in the kept rows; rows are clamped
 *     to M_capacity.
 *   max_seqlen: host upper bound on any cu_kept[b+1] - cu_kept[b] (sizes the grid;
 *     longer sequences set TG_DEV_BAD_SEQLENS).
 *   tau, beta [host] fp32 [H_q]; tau > 0 finite, beta >= 0 finite.
 *   O [device] bf16 [M, H_q, d_h].   status [device] int32 word.
 *   Shapes: d_h == 128 or 64, H_q % H_kv == 0, H_q <= 128; else TG_ERR_UNSUPPORTED.
 *   Compute: bf16 tcgen05 MMA, fp32 softmax and accumulation.
 */
TG_API tg_status tg_gated_attention(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                             const float *g, int32_t H_g, const int32_t *cu_kept, int32_t B,
                             int32_t M_capacity, int32_t max_seqlen, int32_t H_q, int32_t H_kv,
                             int32_t d_h, const float *tau, const float *beta, uint16_t *O,
                             int32_t *status, tg_stream_t stream);

/*
 * tg_gated_attention_workspace_size — bytes of device workspace tg_gated_attention_ws needs for
 *   this shape on the current device (0 when the launch would not split its key ranges).
 *   Arguments as tg_gated_attention. Invalid shapes give 0.
 */
TG_API size_t tg_gated_attention_workspace_size(int32_t B, int32_t max_seqlen, int32_t H_q, int32_t H_kv,
                                                int32_t d_h);

/*
 * tg_gated_attention_ws — tg_gated_attention (deep dive section 3.2, Eqs. (5) and (8)) with a
 *   caller workspace, used when one CTA per 128-row query tile would leave SMs idle (short kept
 *   sequences: small budgets K). Each query tile's causal key range is then cut into chunks of
 *   key tiles, one CTA each; a chunk writes its unnormalised fp32 partial output and its row
 *   statistics (reference max, sum of weights) to the workspace, and the last chunk of the tile
 *   to finish adds the chunks' parts in chunk order (so the result does not depend on which
 *   chunk finishes last) and writes O. Results match tg_gated_attention within rounding.
 *   workspace [device] of workspace_bytes >= tg_gated_attention_workspace_size(...) for the
 *     same B, max_seqlen, H_q, H_kv, d_h, 256-byte aligned; may be NULL (with 0 bytes) when
 *     that size is 0. Its first bytes are arrival counters: the workspace must be zero-filled
 *     before its first use, and every call that completes leaves them zero again. After a call
 *     that reported TG_DEV_TIMEOUT, zero it again. Calls that share a workspace must not run
 *     concurrently. Too small or misaligned: TG_ERR_INVALID_ARG.
 *   Other arguments, layouts and errors as tg_gated_attention.
 */
TG_API tg_status tg_gated_attention_ws(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                                const float *g, int32_t H_g, const int32_t *cu_kept, int32_t B,
                                int32_t M_capacity, int32_t max_seqlen, int32_t H_q, int32_t H_kv,
                                int32_t d_h, const float *tau, const float *beta, uint16_t *O,
                                void *workspace, size_t workspace_bytes, int32_t *status,
                                tg_stream_t stream);

/*
 * tg_gated_attention_noalloc — tg_gated_attention_ws without a caller workspace, for callers that
 *   cannot allocate device memory: code running while another allocator owns the device's memory
 *   (a framework's caching pool, a serving runtime that reserves all memory up front), or code
 *   whose hot path must not allocate. It has no counterpart in the TokenGate pages: it only moves
 *   the split launch's scratch from the caller into the library.
 *   The scratch is a fixed 16 MiB array in device memory that every GPU loading this library
 *   holds until the process exits; the call itself allocates and frees nothing. A shape whose
 *   split needs more than 16 MiB (tg_gated_attention_workspace_size above it) returns
 *   TG_ERR_UNSUPPORTED and launches nothing; use tg_gated_attention_ws for it.
 *   The first call on a device looks up the array's device address; make that first call
 *   before any stream capture on that device. Every call clears the array's arrival counters on
 *   the stream before its kernel. All calls on a device share the one array: calls whose
 *   kernels overlap on the GPU (other streams, other host threads) race on it and must not run
 *   concurrently.
 *   Arguments, layouts, results and other errors as tg_gated_attention.
 */
TG_API tg_status tg_gated_attention_noalloc(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                                            const float *g, int32_t H_g, const int32_t *cu_kept, int32_t B,
                                            int32_t M_capacity, int32_t max_seqlen, int32_t H_q, int32_t H_kv,
                                            int32_t d_h, const float *tau, const float *beta, uint16_t *O,
                                            int32_t *status, tg_stream_t stream);

/*
 * tg_gated_attention_lse — tg_gated_attention that also writes, for every kept row i and query
 *   head h, lse[i * H_q + h] = ln sum_{j <= i} exp(tau_h q_i.k_j / sqrt(d_h) + beta_h ln g_j)
 *   (-inf when every key has zero weight): what the backward needs to rebuild P.
 *   lse [device] fp32 [M_capacity, H_q]. Other arguments as tg_gated_attention.
 */
TG_API tg_status tg_gated_attention_lse(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                                 const float *g, int32_t H_g, const int32_t *cu_kept, int32_t B,
                                 int32_t M_capacity, int32_t max_seqlen, int32_t H_q, int32_t H_kv,
                                 int32_t d_h, const float *tau, const float *beta, uint16_t *O,
                                 float *lse, int32_t *status, tg_stream_t stream);

/*
 * tg_gated_attention_bwd — gradients of a loss through tg_gated_attention (deep dive section
 *   3.2: the gate score reaches the loss only through the attention bias; section 3.1: the top-K
 *   choice itself has no gradient). With P_ij = exp(x_ij - lse_i), dX_ij = P_ij (dO_i.v_j - dO_i.o_i):
 *     dQ [device] fp32 [M, H_q, d_h]  = tau_h / sqrt(d_h) sum_j dX_ij k_j
 *     dK, dV [device] fp32 [M, H_kv, d_h]: sums over the query heads of each GQA group
 *     dbias [device] fp32 [M, H_q]: sum_i dX_ij, the gradient w.r.t. the head-h bias
 *       beta_h ln g_j (so dL/d ln g_j = sum_h beta_h dbias[j, h]).
 *   O, dO [device] bf16 [M, H_q, d_h] (the forward's output and the incoming gradient);
 *   lse from tg_gated_attention_lse. Outputs are overwritten for rows < min(cu_kept[B], M_capacity).
 *   dQ also serves as the call's workspace: D_i = dO_i . o_i is kept in dQ[i, h, 0] until the
 *   final pass writes dQ, so the library allocates nothing.
 *   Compute: tcgen05 MMAs (bf16 operands, fp32 accumulation; P and c_h dX enter the products
 *   rounded to bf16), fp32 elementwise. Deterministic (fixed-order sums, no atomics).
 *   Other arguments as tg_gated_attention.
 */
TG_API tg_status tg_gated_attention_bwd(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                                 const float *g, int32_t H_g, const uint16_t *O, const uint16_t *dO,
                                 const float *lse, const int32_t *cu_kept, int32_t B,
                                 int32_t M_capacity, int32_t max_seqlen, int32_t H_q, int32_t H_kv,
                                 int32_t d_h, const float *tau, const float *beta, float *dQ,
                                 float *dK, float *dV, float *dbias, int32_t *status,
                                 tg_stream_t stream);

/*
 * tg_gate_score_grad — carry the attention bias gradient back to the gate scores:
 *   ds[kept_idx[m], c] = (1 - g_kept[m, c]) * sum over the query heads h that read gate head c
 *   of beta_h dbias[m, h], for m < min(cu_kept[B], capacity) (d ln g / ds = 1 - g for
 *   g = sigmoid(s); non-prunable rows have g = 1, so they get 0). With H_g = 1 every head
 *   reads the one gate. Rows that were not kept are not written: the caller zeroes
 *   ds [device] fp32 [T_total, H_g].
 *   dbias [device] fp32 [capacity, H_q]; beta [host] fp32 [H_q];
 *   g_kept [device] fp32 [capacity, H_g]; 1 <= H_g <= 16, H_q % H_g == 0.
 */
TG_API tg_status tg_gate_score_grad(const float *dbias, const float *beta, const float *g_kept, int32_t H_g,
                             const int32_t *kept_idx, const int32_t *cu_kept, int32_t B,
                             int32_t capacity, int32_t H_q, int32_t T_total, float *ds,
                             tg_stream_t stream);

/*
 * tg_gate_prune_layer — tg_gate_score, tg_topk_select and tg_gather_kept enqueued back to
 *   back on one stream (the deep dive's section 3.4 prune path: score, clamp, select, keep
 *   indices, slice hidden states, gather positions). Arguments as in the three calls;
 *   s_out and g_out are required here (they are the intermediate buffers).
 */
TG_API tg_status tg_gate_prune_layer(const uint16_t *h, const int32_t *pos, const uint8_t *instr_mask,
                              const int32_t *cu_seqlens, int32_t B, int32_t T_total, int32_t d,
                              const uint16_t *W1, const float *b1, const uint16_t *w2, float b2,
                              int32_t d_g, int32_t K, float *s_out, float *g_out,
                              int32_t *kept_idx, int32_t capacity, int32_t *cu_kept,
                              uint16_t *h_kept, int32_t *pos_kept, float *g_kept,
                              int32_t *status, tg_stream_t stream);

/*
 * tg_gate_prune_layer_heads — the prune path with per-head gates: tg_gate_score_heads, then
 *   tg_topk_select on the head mean s_sel, then tg_gather_kept of the H_g gate values per
 *   kept row (g_kept [device] fp32 [capacity, H_g]). Arguments as in those calls; s_heads,
 *   g_heads and s_sel are required here.
 */
TG_API tg_status tg_gate_prune_layer_heads(const uint16_t *h, const int32_t *pos, const uint8_t *instr_mask,
                                    const int32_t *cu_seqlens, int32_t B, int32_t T_total, int32_t d,
                                    const uint16_t *W1, const float *b1, const uint16_t *W2, const float *b2,
                                    int32_t d_g, int32_t H_g, int32_t K, float *s_heads, float *g_heads,
                                    float *s_sel, int32_t *kept_idx, int32_t capacity, int32_t *cu_kept,
                                    uint16_t *h_kept, int32_t *pos_kept, float *g_kept, int32_t *status,
                                    tg_stream_t stream);

/*
 * tg_two_budget_prune_layer — the packed two-budget forward of training (deep dive section 3.3,
 *   Eq. (9): K_full = |P| and K_prune ~ LogUniform(1, |P|/2), "packed into one variable-length
 *   call", phase 1 evaluated once). Scores once, then writes ONE keep list of 2B sequences:
 *   sequences 0..B-1 are the full budget (every row: the identity) and sequences B..2B-1 the
 *   K_prune selection of the same inputs, placed after them. cu_packed [device] int32 [2B+1]:
 *   cu_packed[0..B] = cu_seqlens, cu_packed[B + b + 1] = T_total + (rows kept in the pruned
 *   sequences 0..b). kept_idx / h_kept / pos_kept / g_kept follow the packed list, so one
 *   tg_gated_attention call over (cu_packed, 2B sequences) serves both budgets.
 *   capacity >= T_total is required; 2 * T_total is always enough. The caller draws K_prune.
 *   Other arguments and errors as tg_gate_prune_layer; 1 <= B <= 512.
 */
TG_API tg_status tg_two_budget_prune_layer(const uint16_t *h, const int32_t *pos, const uint8_t *instr_mask,
                                    const int32_t *cu_seqlens, int32_t B, int32_t T_total, int32_t d,
                                    const uint16_t *W1, const float *b1, const uint16_t *w2, float b2,
                                    int32_t d_g, int32_t K_prune, float *s_out, float *g_out,
                                    int32_t *kept_idx, int32_t capacity, int32_t *cu_packed,
                                    uint16_t *h_kept, int32_t *pos_kept, float *g_kept,
                                    int32_t *status, tg_stream_t stream);

/*
 * tg_apply_rope — rotate Q or K rows in place at their original position ids (rotate-half
 *   form, inv_freq_i = theta^(-2i/d_h)); the deep dive (section 3.4) keeps the original
 *   position ids for the kept tokens.
 *   X [device] bf16 [capacity, H, d_h];  pos [device] int32 [capacity].
 *   cu_kept [device] int32 [B+1] or NULL: when given, only rows < min(cu_kept[B], capacity)
 *   are touched; when NULL, all `capacity` rows are.
 *   d_h even, d_h <= 256; theta > 0.
 */
TG_API tg_status tg_apply_rope(uint16_t *X, const int32_t *pos, const int32_t *cu_kept, int32_t B,
                        int32_t capacity, int32_t H, int32_t d_h, float theta,
                        tg_stream_t stream);

/*
 * tg_normalize_scores — sequence-axis RMS normalisation of the gate scores (deep dive section
 *   3.1, Eq. (3)): b_j = s_j / sqrt(mean over the sequence's prunable rows of s^2 + eps), and
 *   b_j = 0 on non-prunable rows. A sequence without prunable rows gets b = 0. The order of
 *   the prunable scores is unchanged, so top-K may select from s or from b alike.
 *   s [device] fp32 [T_total, H_g] (as written by tg_gate_score / tg_gate_score_heads); each
 *   gate head is normalised on its own. instr_mask [device] uint8 or NULL;
 *   cu_seqlens [device] int32 [B+1]; eps: host, finite, >= 0 (the pages give none; 1e-6 is the
 *   usual choice). b_out [device] fp32 [T_total, H_g].
 *   b_sel [device] fp32 [T_total] or NULL: with H_g > 1, the row mean of the normalised heads
 *   (the uniform head aggregation that top-K ranks; 0 on non-prunable rows). Not written when
 *   H_g = 1 (b_out itself is then the ranking).
 *   status [device] int32 word (TG_DEV_BAD_SEQLENS).
 *   Limits: 1 <= B <= 1024, 1 <= H_g <= 16. The per-sequence sums run in a fixed order
 *   (deterministic).
 */
TG_API tg_status tg_normalize_scores(const float *s, int32_t H_g, const uint8_t *instr_mask,
                              const int32_t *cu_seqlens, int32_t B, int32_t T_total, float eps,
                              float *b_out, float *b_sel, int32_t *status, tg_stream_t stream);

/*
 * tg_gated_attention_eq8 — the operative token-gated attention of the deep dive, section 3.2,
 *   Eq. (8), with the pruning-ratio temperature of Eq. (7):
 *     o_i = sum_{j <= i} softmax_j[ tau_i (q_i.k_j / sqrt(d_h) + gain_h b_j) ] v_j,
 *     tau_i = temp_h ln(m_i) / ln(max(2, p_i)),
 *   m_i = number of retained keys query i sees (its index in the kept sequence + 1),
 *   p_i = number of positions it originally saw (its original position id + 1).
 *   gain_h = softplus(gamma_h) and temp_h = softplus(sigma_h) are passed already transformed.
 *   b   [device] fp32 [M, H_g]: normalised scores of the kept rows (tg_normalize_scores,
 *       gathered by tg_gather_kept), or NULL for no score bias; query head h reads gate head
 *       h / (H_q / H_g) (1 <= H_g <= 16, H_q % H_g == 0; pass 1 when b is NULL).
 *   pos [device] int32 [M]: original position ids of the kept rows (tg_gather_kept's pos_kept).
 *   gain, temp [host] fp32 [H_q], finite and >= 0.
 *   Other arguments, layouts, shapes and errors as tg_gated_attention.
 */
TG_API tg_status tg_gated_attention_eq8(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                                 const float *b, int32_t H_g, const int32_t *pos, const int32_t *cu_kept,
                                 int32_t B, int32_t M_capacity, int32_t max_seqlen, int32_t H_q,
                                 int32_t H_kv, int32_t d_h, const float *gain, const float *temp,
                                 uint16_t *O, int32_t *status, tg_stream_t stream);

/*
 * tg_read_device_status — synchronise `stream`, copy the device status word to *out and
 *   translate it: 0 -> TG_OK, TG_DEV_TIMEOUT -> TG_ERR_DEVICE_TIMEOUT, TG_DEV_CAPACITY ->
 *   TG_ERR_CAPACITY, any other bit -> TG_ERR_DEVICE. *out receives the raw bits.
 */
TG_API tg_status tg_read_device_status(const int32_t *status, int32_t *out, tg_stream_t stream);

/*
 * tg_set_wait_limit_ns — upper bound, in nanoseconds of device time, on any single
 *   pipeline wait inside the tensor-core kernels (default 2e9, i.e. two seconds). A wait
 *   that runs past it sets TG_DEV_TIMEOUT, drains the copies it started and returns.
 *   0 restores the default. Process-wide; takes effect for later launches.
 */
TG_API tg_status tg_set_wait_limit_ns(uint64_t limit_ns);

/*
 * tg_set_test_withhold — failure-injection hook for tests of the bounded waits above (no
 *   counterpart in the TokenGate pages). While a bit is set, the matching kernel's copy
 *   producer issues none of its loads, so the consumers' waits run out after the wait limit;
 *   the kernel sets TG_DEV_TIMEOUT, frees its tensor memory and returns, and the CUDA context
 *   stays usable. Nothing faults or hangs. Bits: TG_WITHHOLD_GATE_SCORE, TG_WITHHOLD_ATTENTION,
 *   TG_WITHHOLD_BACKWARD (the dK/dV and dQ passes of tg_gated_attention_bwd);
 *   TG_WITHHOLD_GATE_SCORE_PEER (only the gate-score CTAs of odd cluster rank withhold theirs,
 *   so every CTA pair loses one half of each stage while the other half lands);
 *   0 (the default) clears them. Any other bit is TG_ERR_INVALID_ARG. Process-wide; takes
 *   effect for later launches.
 */
enum {
  TG_WITHHOLD_GATE_SCORE = 1 << 0,
  TG_WITHHOLD_ATTENTION = 1 << 1,
  TG_WITHHOLD_BACKWARD = 1 << 2,
  TG_WITHHOLD_GATE_SCORE_PEER = 1 << 3
};
TG_API tg_status tg_set_test_withhold(int32_t mask);

#ifdef __cplusplus
}
#endif

#endif /* TOKENGATE_H_ */
