// tg_attention.cu — token-gated causal GQA attention over the kept tokens (TokenGate deep
// dive, section 3.2: Eq. (5), alpha_ij proportional to exp(z_ij) g_j; Eq. (8) with the gate
// as a per-key, per-head bias inside the softmax and a temperature on the logits).
//
//   o_i = sum_{j<=i} softmax_j( tau_h * q_i.k_j / sqrt(d_h) + beta_h * ln g_j ) v_j
//
// Computed in base 2: x_ij = s_ij * (tau_h log2(e) / sqrt(d_h)) + beta_h log2(g_j), p = 2^(x - m).
//
// One CTA handles one 128-row query tile of one sequence for TWO query heads that read the
// same kv head (a GQA pair), so every K/V tile brought in by TMA feeds two Q tiles. Tensor
// memory (512 columns) holds S_0, S_1 (fp32 128x128 each; P_t is written back over S_t as
// packed bf16) and the output accumulators O_0, O_1 (fp32 128 x d_h).
// Warp roles (12 warps):
//   warp 0       TMA producer: Q tiles once, then the K/V ring (kStages deep)
//   warp 1       tensor-memory owner and MMA issuer:  S_t = Q_t K^T ; O_t += P_t V (the warp runs
//                converged and one elected lane issues, which keeps the operands warp-uniform)
//   warp 2       bias producer: beta_h * log2(g_j) of each K/V tile's 128 keys, both heads,
//                into a shared-memory ring that follows the K/V stages. The gate may be per
//                head (section 3.4: a per-head bias): g is [M, H_g] and query head h reads
//                gate head h / (H_q / H_g)
//   warps 4-7    softmax + correction + epilogue for Q tile 0 (thread = query row = TMEM lane)
//   warps 8-11   the same for Q tile 1
// Online softmax with a lazily updated running max: the reference max m only moves when the
// tile max exceeds it by more than 8 (log2 units), so the O rescale (a TMEM read-modify-write)
// is rare; the result is exact either way because O and l share the same reference. The
// softmax runs on packed fp32 pairs (fma/add .f32x2) with 3-input max, and only the diagonal
// key tile carries the causal mask.
#include <algorithm>
#include <mutex>

#include "tg_common.cuh"

namespace {

constexpr int kBlockM = 128;      // query rows per tile
constexpr int kBlockN = 128;      // keys per KV tile
constexpr int kThreads = 384;
constexpr float kRescaleThreshold = 8.0f;
constexpr int kMaxHeads = 128;
constexpr int kMaxChunkItems = 256;  // (query tile, key chunk) entries of a split launch
constexpr int kMaxChunks = 3;        // chunks of one query tile in a split launch
// Split only when the heaviest query tile walks at least this many key tiles: below that, the
// extra arrival and combine (about two key steps) cost more than the shorter walk saves.
constexpr int kMinSplitSteps = 6;

template <int D>
struct AttnCfg {
  static constexpr int kHalves = D / 64;                    // 128-byte swizzle atoms per row
  static constexpr uint32_t kTileBytes = 128u * D * 2u;     // one 128-row bf16 tile
  static constexpr int kStages = D == 128 ? 2 : 3;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffK = 2 * kTileBytes;
  static constexpr uint32_t kOffV = kOffK + kStages * kTileBytes;
  static constexpr uint32_t kOffBias = kOffV + kStages * kTileBytes;       // [stage][2 heads][128] f32
  static constexpr uint32_t kOffBar = kOffBias + kStages * 2 * 128 * 4;
  static constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 384;
};

// Two forms of the score bias and temperature (TokenGate deep dive, section 3.2):
//   kLogGate: logit = tau_h q.k / sqrt(d_h) + beta_h ln g_j                 (Eq. (5) in log form)
//   kEq8:     logit = tau_i (q.k / sqrt(d_h) + gain_h b_j),                  (Eq. (8))
//             tau_i = temp_h ln(m_i) / ln(max(2, p_i))                        (Eq. (7))
//             with m_i = i - start + 1 retained keys, p_i = pos_i + 1 original positions.
enum { kLogGate = 0, kEq8 = 1 };

struct AttnParams {
  const float *g;            // kLogGate: gate values g_j; kEq8: normalised scores b_j (or NULL)
  int32_t g_cols, g_group;   // gate heads per row (H_g); query heads per gate head (H_q / H_g)
  const int32_t *pos;        // kEq8: original position ids of the kept rows
  const int32_t *cu_kept;
  int32_t B, M_cap, max_seqlen, H_q, H_kv, group, heads_per_cta, pairs, n_qt_max;
  uint16_t *O;
  float *lse;  // optional [M, H_q]: natural-log log-sum-exp of each row's logits (for the backward)
  int32_t *status;
  uint64_t wait_limit, drain_limit;
  int32_t withhold;  // test hook: issue no loads, so the consumers' waits run out
  // Split key range (a launch that would leave SMs idle): query tile tq's key tiles 0..tq are cut
  // into chunks of `chunk` tiles, one CTA each. A chunk writes its unnormalised fp32 partial O
  // and its (reference max, row sum) to a workspace slot; the last chunk of a tile to finish
  // (an arrival counter per tile) combines the slots in chunk order and writes O. Each counter
  // is reset to 0 by the combining CTA, so a workspace that starts zeroed stays reusable.
  int32_t split;       // 0: one CTA per query tile
  int32_t chunk;       // key tiles per chunk
  int32_t n_u;         // (query tile, chunk) entries per (sequence, head pair)
  int32_t *ws_count;   // [B * pairs * n_qt_max] arrival counters
  float *ws_part;      // [B * pairs * n_u] slots of SlotFloats<D>() floats
  uint32_t u_tab[kMaxChunkItems];  // entry -> tq | chunk index << 16, heaviest first
  float scale_log2[kMaxHeads];  // kLogGate: tau_h * log2(e) / sqrt(d_h); kEq8: temp_h
  float beta[kMaxHeads];        // kLogGate: beta_h; kEq8: gain_h * log2(e)
};

// One workspace slot of a split launch: O as [2 heads][D / 4 column blocks][128 rows] float4
// (unnormalised fp32), then (m, l) as [2 heads][128 rows] float2.
template <int D>
__host__ __device__ constexpr size_t slot_floats() {
  return static_cast<size_t>(2) * 128 * D + 2 * 128 * 2;
}

// Slots of query tiles 0..tq-1 (tile t has ceil((t + 1) / chunk) chunks).
__host__ __device__ inline int chunk_slot_base(int tq, int chunk) {
  int s = 0;
  for (int t = 0; t < tq; ++t) s += (t + chunk) / chunk;
  return s;
}

__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// log2 of a gate value; a subnormal gate keeps its own weight g^beta (see tg::log2_gate)
__device__ __forceinline__ float lg2(float x) { return tg::log2_gate(x); }

// Packed fp32 pairs (Blackwell .f32x2 arithmetic).
__device__ __forceinline__ uint64_t f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float &a, float &b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

template <int D, int MODE, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    gated_attention_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v,
                           const __grid_constant__ AttnParams p) {
  using C = AttnCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = smem + C::kOffQ;
  uint8_t *sK = smem + C::kOffK;
  uint8_t *sV = smem + C::kOffV;
  float *sBias = reinterpret_cast<float *>(smem + C::kOffBias);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
  uint64_t *q_full = bars;
  uint64_t *kv_full = bars + 1;
  uint64_t *kv_empty = kv_full + C::kStages;
  uint64_t *s_full = kv_empty + C::kStages;  // [2]
  uint64_t *p_full = s_full + 2;             // [2]
  uint64_t *o_final = p_full + 2;            // [2]
  uint64_t *pv_done = o_final + 2;           // [2]
  uint64_t *bias_full = pv_done + 2;         // [kStages]
  uint64_t *drain = bias_full + C::kStages;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  int32_t *abort_flag = reinterpret_cast<int32_t *>(tmem_slot + 1);
  int32_t *n_issued = abort_flag + 1;
  int32_t *n_consumed = abort_flag + 2;
  int32_t *q_issued = abort_flag + 3;
  volatile int32_t *vabort = abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  tg::pdl_wait();
  tg::pdl_launch_dependents();
  // ---- work item: heaviest (last) query tiles first ----
  const int item = blockIdx.x;
  const int hp = item % p.pairs;
  const int rest = item / p.pairs;
  const int b = rest % p.B;
  int tq, chunk_id = 0;
  if (SPLIT) {
    const uint32_t e = p.u_tab[rest / p.B];
    tq = static_cast<int>(e & 0xFFFFu);
    chunk_id = static_cast<int>(e >> 16);
  } else {
    tq = p.n_qt_max - 1 - rest / p.B;
  }
  int seq_start = p.cu_kept[b];
  int seq_end = p.cu_kept[b + 1];
  if (seq_start < 0 || seq_end < seq_start || seq_end - seq_start > p.max_seqlen) {
    if (threadIdx.x == 0 && tq == p.n_qt_max - 1 && hp == 0 && chunk_id == 0) tg::report(p.status, TG_DEV_BAD_SEQLENS);
    return;
  }
  seq_start = min(seq_start, p.M_cap);
  seq_end = min(seq_end, p.M_cap);
  const int seq_len = seq_end - seq_start;
  const int q0 = tq * kBlockM;
  if (q0 >= seq_len) return;  // uniform for the CTA
  // causal: key tiles 0..tq, or this CTA's chunk j0 .. j0 + n_kv - 1 of them
  const int j0 = SPLIT ? chunk_id * p.chunk : 0;
  const int n_kv = SPLIT ? min(p.chunk, tq + 1 - j0) : tq + 1;
  const int n_chunks = SPLIT ? (tq + p.chunk) / p.chunk : 1;
  const int h0 = hp * p.heads_per_cta;
  const int kvh = h0 / p.group;
  const int n_tiles = p.heads_per_cta;  // Q tiles in this CTA (1 or 2)

  if (threadIdx.x == 0) {
    tg::mbar_init(q_full, 1);
    for (int i = 0; i < C::kStages; ++i) {
      tg::mbar_init(&kv_full[i], 1);
      tg::mbar_init(&kv_empty[i], 1);
      tg::mbar_init(&bias_full[i], 32);
    }
    for (int t = 0; t < 2; ++t) {
      tg::mbar_init(&s_full[t], 1);
      tg::mbar_init(&p_full[t], 128);
      tg::mbar_init(&o_final[t], 1);
      tg::mbar_init(&pv_done[t], 1);
    }
    tg::mbar_init(drain, 1);
    *abort_flag = 0;
    *n_issued = 0;
    *n_consumed = 0;
    *q_issued = 0;
    tg::fence_mbar_init();
    tg::prefetch_tensormap(&tm_q);
    tg::prefetch_tensormap(&tm_k);
    tg::prefetch_tensormap(&tm_v);
  }
  if (warp == 1) {
    tg::tmem_alloc(tmem_slot, 512);
    tg::tmem_relinquish();
  }
  tg::tc_fence_before();
  __syncthreads();
  tg::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0 && !p.withhold) {
      // ---------------- TMA producer ----------------
      *q_issued = 1;
      tg::mbar_arrive_expect_tx(q_full, n_tiles * C::kTileBytes);
      for (int t = 0; t < n_tiles; ++t)
        for (int hf = 0; hf < C::kHalves; ++hf)
          tg::tma_load_3d(sQ + t * C::kTileBytes + hf * 16384, &tm_q, q_full, hf * 64, h0 + t,
                          seq_start + q0);
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % C::kStages;
        const uint32_t ph = (j / C::kStages) & 1;
        if (!tg::mbar_wait(&kv_empty[st], ph ^ 1u, vabort, p.wait_limit)) {
          *vabort = 1;
          break;
        }
        tg::mbar_arrive_expect_tx(&kv_full[st], 2 * C::kTileBytes);
        for (int hf = 0; hf < C::kHalves; ++hf) {
          tg::tma_load_3d(sK + st * C::kTileBytes + hf * 16384, &tm_k, &kv_full[st], hf * 64, kvh,
                          seq_start + (j0 + j) * kBlockN);
          tg::tma_load_3d(sV + st * C::kTileBytes + hf * 16384, &tm_v, &kv_full[st], hf * 64, kvh,
                          seq_start + (j0 + j) * kBlockN);
        }
        issued = j + 1;
      }
      *n_issued = issued;
    }
  } else if (warp == 1) {
    {
      // ---------------- MMA issuer: the whole warp runs the loop, one elected lane issues ----------------
      const uint32_t idesc_s = tg::idesc_bf16_f32(kBlockM, kBlockN);        // Q K^T, both K-major
      const uint32_t idesc_o = tg::idesc_bf16_f32(kBlockM, D, 0, 1);        // P V, V MN-major
      const uint32_t colS[2] = {C::kColS0, C::kColS1};
      const uint32_t colO[2] = {C::kColO0, C::kColO1};
      bool ok = __all_sync(0xFFFFFFFFu, tg::mbar_wait(q_full, 0, vabort, p.wait_limit));
      int consumed = 0;
      // descriptors of each operand buffer, built once; a K-step adds its byte offset / 16
      // (buffers of one kind are contiguous, so buffer i is the first one's descriptor + i * tile / 16)
      const uint64_t dq0 = tg::smem_desc(tg::smem_u32(sQ), 16, 1024, tg::kSwz128);
      const uint64_t dk0 = tg::smem_desc(tg::smem_u32(sK), 16, 1024, tg::kSwz128);
      const uint64_t dv0 = tg::smem_desc(tg::smem_u32(sV), 16384, 1024, tg::kSwz128);
      constexpr uint32_t kTile16 = C::kTileBytes >> 4;
      auto issue_s = [&](int t, int st) {
        const uint64_t qd = dq0 + t * kTile16, kd = dk0 + st * kTile16;
        const uint32_t dst = tmem + colS[t];
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off16 = ((k / 4) * 16384 + (k % 4) * 32) >> 4;
          tg::mma_bf16_ss_elect(dst, qd + off16, kd + off16, idesc_s, k != 0);
        }
        tg::mma_commit_elect(&s_full[t]);
      };
      auto issue_pv = [&](int t, int st, bool first) {
        const uint64_t vd = dv0 + st * kTile16;
        const uint32_t dst = tmem + colO[t], src = tmem + colS[t];
#pragma unroll
        for (int k = 0; k < kBlockN / 16; ++k) {
          // keys 16k..16k+15: 16 rows of 128 B in every d-half; d-halves 16 KB apart
          tg::mma_bf16_ts_elect(dst, src + k * 8, vd + ((k * 2048) >> 4), idesc_o, !(first && k == 0));
        }
      };
      if (ok) {
        if (!__all_sync(0xFFFFFFFFu, tg::mbar_wait(&kv_full[0], 0, vabort, p.wait_limit))) ok = false;
      }
      if (ok) {
        tg::tc_fence_after();
        for (int t = 0; t < n_tiles; ++t) issue_s(t, 0);
        // Per step j and tile t: PV_t(j) once P_t(j) is in tensor memory; then S_t(j+1), but
        // only after PV_t(j) has finished reading P_t(j), whose columns S_t(j+1) overwrites.
        for (int j = 0; j < n_kv && ok; ++j) {
          const int st = j % C::kStages;
          const bool has_next = j + 1 < n_kv;
          const int st_n = (j + 1) % C::kStages;
          for (int t = 0; t < n_tiles && ok; ++t) {
            if (!__all_sync(0xFFFFFFFFu, tg::mbar_wait(&p_full[t], j & 1, vabort, p.wait_limit))) {
              ok = false;
              break;
            }
            tg::tc_fence_after();
            issue_pv(t, st, j == 0);
            tg::mma_commit_elect(has_next ? &pv_done[t] : &o_final[t]);
            if (t == n_tiles - 1) {
              tg::mma_commit_elect(&kv_empty[st]);
              consumed = j + 1;
            }
            if (has_next) {
              if (t == 0 &&
                  !__all_sync(0xFFFFFFFFu, tg::mbar_wait(&kv_full[st_n], ((j + 1) / C::kStages) & 1, vabort,
                                                         p.wait_limit))) {
                ok = false;
                break;
              }
              if (!__all_sync(0xFFFFFFFFu, tg::mbar_wait(&pv_done[t], j & 1, vabort, p.wait_limit))) {
                ok = false;
                break;
              }
              tg::tc_fence_after();
              issue_s(t, st_n);
            }
          }
        }
      }
      if (lane == 0) *n_consumed = consumed;
      if (!ok) {
        *vabort = 1;
        tg::mma_commit_elect(drain);
        volatile int32_t never = 0;
        tg::mbar_wait(drain, 0, &never, p.drain_limit);
      }
    }
  } else if (warp == 2) {
    // ---------------- bias producer: the per-key bias of each K/V tile, both heads ----------------
    if (p.g != nullptr) {
      const float beta0 = p.beta[h0];
      const float beta1 = n_tiles > 1 ? p.beta[h0 + 1] : 0.0f;
      // per-head gates: query head h reads gate head h / g_group of its key's row
      const int col0 = h0 / p.g_group;
      const int col1 = n_tiles > 1 ? (h0 + 1) / p.g_group : col0;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % C::kStages;
        const uint32_t ph = (j / C::kStages) & 1;
        // the stage is free once both tiles' PV of step j - kStages has completed (the same
        // barrier that frees the K/V stage); by then both softmax warpgroups are done with it
        if (!tg::mbar_wait(&kv_empty[st], ph ^ 1u, vabort, p.wait_limit)) {
          *vabort = 1;
          break;
        }
        float *dst = sBias + st * 256;
        float gv0[4], gv1[4];
        const float pad = MODE == kEq8 ? 0.0f : 1.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int k = (j0 + j) * kBlockN + lane * 4 + i;
          const size_t row = static_cast<size_t>(seq_start + k) * p.g_cols;
          gv0[i] = k < seq_len ? p.g[row + col0] : pad;
          gv1[i] = col1 == col0 ? gv0[i] : (k < seq_len ? p.g[row + col1] : pad);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          // kLogGate: beta_h log2(g_j) (beta = 0 means g^0 = 1, a zero bias even where g = 0);
          // kEq8: gain_h log2(e) b_j, the log2-unit score bias before the row's temperature
          const float v0 = MODE == kEq8 ? gv0[i] : lg2(gv0[i]);
          const float v1 = col1 == col0 ? v0 : (MODE == kEq8 ? gv1[i] : lg2(gv1[i]));
          dst[lane * 4 + i] = beta0 == 0.0f ? 0.0f : beta0 * v0;
          dst[128 + lane * 4 + i] = beta1 == 0.0f ? 0.0f : beta1 * v1;
        }
        tg::mbar_arrive(&bias_full[st]);
      }
    }
  } else if (warp >= 4) {
    // ---------------- softmax / correction / epilogue ----------------
    const int t = (warp - 4) >> 2;          // Q tile 0 (warps 4-7) or 1 (warps 8-11)
    const int wq = warp & 3;                 // TMEM lane quarter
    const int r = wq * 32 + lane;            // query row within the tile
    float m_ref = -INFINITY;  // reference max (log2 units)
    float l = 0.0f;           // row sum relative to it
    if (t < n_tiles) {
      const int h = h0 + t;
      const float scale = p.scale_log2[h];
      const bool use_bias = p.g != nullptr;  // beta = 0 arrives as a zero bias
      const uint32_t colS = t == 0 ? C::kColS0 : C::kColS1;
      const uint32_t colO = t == 0 ? C::kColO0 : C::kColO1;
      const uint32_t lane_addr = tmem + (static_cast<uint32_t>(wq * 32) << 16);
      // kEq8: this row's temperature (Eq. (7)); rows past the sequence end are never stored
      float tau_row = 1.0f;
      if (MODE == kEq8) {
        const int i_local = q0 + r;  // index of the query in its kept sequence
        if (i_local < seq_len) {
          const int m_i = i_local + 1;
          const int p_i = p.pos[seq_start + i_local] + 1;
          tau_row = scale * (logf(static_cast<float>(m_i)) / logf(static_cast<float>(max(2, p_i))));
        }
      }
      // kLogGate: x = s * scale + bias.  kEq8: x = tau_i * (s * log2(e) / sqrt(d_h) + bias)
      const float c1 = 1.4426950408889634f / sqrtf(static_cast<float>(D));
      const float s_mul = MODE == kEq8 ? (use_bias ? c1 : c1 * tau_row) : scale;
      const uint64_t scale2 = f2(s_mul, s_mul);
      const uint64_t tau2 = f2(tau_row, tau_row);
      bool ok = true;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % C::kStages;
        bool w = tg::mbar_wait(&s_full[t], j & 1, vabort, p.wait_limit);
        if (use_bias) w = w && tg::mbar_wait(&bias_full[st], (j / C::kStages) & 1, vabort, p.wait_limit);
        ok = __all_sync(0xFFFFFFFFu, w);  // tcgen05.ld below is warp-collective
        if (!ok) break;
        tg::tc_fence_after();
        // S row (128 fp32) -> logits in log2 units, in place: x = s * scale + bias
        uint32_t x[128];
        tg::tmem_ld_32x32b_x32(lane_addr + colS + 0, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
        tg::tmem_ld_32x32b_x32(lane_addr + colS + 32, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
        tg::tmem_ld_32x32b_x32(lane_addr + colS + 64, *reinterpret_cast<uint32_t(*)[32]>(&x[64]));
        tg::tmem_ld_32x32b_x32(lane_addr + colS + 96, *reinterpret_cast<uint32_t(*)[32]>(&x[96]));
        tg::tmem_ld_wait();
        if (use_bias) {
          const float4 *bias4 = reinterpret_cast<const float4 *>(sBias + st * 256 + t * 128);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float4 bv = bias4[c];
            float a0, a1, a2, a3;
            uint64_t v01 = f2_fma(f2(__uint_as_float(x[4 * c]), __uint_as_float(x[4 * c + 1])), scale2, f2(bv.x, bv.y));
            uint64_t v23 = f2_fma(f2(__uint_as_float(x[4 * c + 2]), __uint_as_float(x[4 * c + 3])), scale2, f2(bv.z, bv.w));
            if (MODE == kEq8) {
              v01 = f2_mul(v01, tau2);
              v23 = f2_mul(v23, tau2);
            }
            f2_split(v01, a0, a1);
            f2_split(v23, a2, a3);
            x[4 * c] = __float_as_uint(a0);
            x[4 * c + 1] = __float_as_uint(a1);
            x[4 * c + 2] = __float_as_uint(a2);
            x[4 * c + 3] = __float_as_uint(a3);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            float a0, a1;
            f2_split(f2_mul(f2(__uint_as_float(x[2 * c]), __uint_as_float(x[2 * c + 1])), scale2), a0, a1);
            x[2 * c] = __float_as_uint(a0);
            x[2 * c + 1] = __float_as_uint(a1);
          }
        }
        if (j0 + j == tq) {
          // diagonal tile: key c is visible to row r only when c <= r
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > r) x[c] = __float_as_uint(-INFINITY);
        }
        // row max over 8 independent chains, then combined
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = fmax3(__uint_as_float(x[i]), __uint_as_float(x[8 + i]), __uint_as_float(x[16 + i]));
#pragma unroll
        for (int c = 24; c < 120; c += 16) {  // columns 24..119, two per chain per step
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = fmax3(mx[i], __uint_as_float(x[c + i]), __uint_as_float(x[c + 8 + i]));
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = fmaxf(mx[i], __uint_as_float(x[120 + i]));  // columns 120..127
        const float tile_max = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
        // lazy max update; rescale O and l only when the max moved by more than the threshold
        float alpha = 1.0f;
        bool rescale = false;
        if (j == 0) {
          m_ref = tile_max;
        } else if (tile_max > m_ref + kRescaleThreshold) {
          alpha = ex2(m_ref - tile_max);
          m_ref = tile_max;
          rescale = true;
        }
        const float m_use = (m_ref == -INFINITY) ? 0.0f : m_ref;
        const uint64_t negm2 = f2(-m_use, -m_use);
        // p = 2^(x - m), packed to bf16 pairs in place (x[c] is dead once pair c/2 is done);
        // the row sum runs on four independent pair accumulators
        uint64_t sum2[4] = {f2(0.0f, 0.0f), f2(0.0f, 0.0f), f2(0.0f, 0.0f), f2(0.0f, 0.0f)};
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          float a, bb;
          f2_split(f2_add(f2(__uint_as_float(x[2 * c]), __uint_as_float(x[2 * c + 1])), negm2), a, bb);
          const float pa = ex2(a), pb = ex2(bb);
          sum2[c & 3] = f2_add(sum2[c & 3], f2(pa, pb));
          x[c] = tg::pack_bf16x2(pa, pb);
        }
        float s_lo, s_hi, t_lo, t_hi;
        f2_split(f2_add(f2_add(sum2[0], sum2[1]), f2_add(sum2[2], sum2[3])), s_lo, s_hi);
        (void)t_lo;
        (void)t_hi;
        l = l * alpha + (s_lo + s_hi);
        if (__any_sync(0xFFFFFFFFu, rescale)) {
          // O_t *= alpha for this row (the PV of step j-1 into O_t has completed: S_t(j) was
          // issued after it, and s_full fired only when every earlier MMA had finished)
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tg::tmem_ld_32x32b_x32(lane_addr + colO + c0, o);
            tg::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tg::tmem_st_32x32b_x32(lane_addr + colO + c0, o);
          }
        }
        // P (bf16 pairs) over the first 64 columns of S_t
        tg::tmem_st_32x32b_x32(lane_addr + colS + 0, *reinterpret_cast<const uint32_t(*)[32]>(&x[0]));
        tg::tmem_st_32x32b_x32(lane_addr + colS + 32, *reinterpret_cast<const uint32_t(*)[32]>(&x[32]));
        tg::tmem_st_wait();
        tg::tc_fence_before();
        tg::mbar_arrive(&p_full[t]);
      }
      // ---- epilogue: O / l -> bf16 rows of O (or this chunk's partial row to its slot) ----
      if (ok) ok = __all_sync(0xFFFFFFFFu, tg::mbar_wait(&o_final[t], 0, vabort, p.wait_limit));
      if (SPLIT && ok && n_chunks > 1) {
        tg::tc_fence_after();
        // unnormalised fp32 O row and (reference max, row sum), both relative to m_use
        const int row = q0 + r;
        float *slot = p.ws_part + (static_cast<size_t>(b * p.pairs + hp) * p.n_u +
                                   chunk_slot_base(tq, p.chunk) + chunk_id) * slot_floats<D>();
        // column-block-major: float4 c4 of row r at [t][c4][r], so a warp's 32 rows are 512
        // contiguous bytes for every store here and every load of the combine
        float4 *opart = reinterpret_cast<float4 *>(slot) + static_cast<size_t>(t) * (D / 4) * 128 + r;
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tg::tmem_ld_32x32b_x32(lane_addr + colO + c0, o);
          tg::tmem_ld_wait();
          if (row < seq_len) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              opart[(c0 / 4 + i) * 128] = make_float4(__uint_as_float(o[4 * i]), __uint_as_float(o[4 * i + 1]),
                                                      __uint_as_float(o[4 * i + 2]), __uint_as_float(o[4 * i + 3]));
          }
        }
        if (row < seq_len)
          *reinterpret_cast<float2 *>(slot + static_cast<size_t>(2) * 128 * D + (t * 128 + r) * 2) =
              make_float2((m_ref == -INFINITY) ? 0.0f : m_ref, l);
      } else if (ok) {
        tg::tc_fence_after();
        const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
        const int row = q0 + r;
        if (p.lse != nullptr && row < seq_len) {
          // x is in log2 units relative to m_ref: ln sum exp = (m + log2 l) ln 2
          const float m_use = (m_ref == -INFINITY) ? 0.0f : m_ref;
          p.lse[static_cast<size_t>(seq_start + row) * p.H_q + h] =
              l > 0.0f ? (m_use + log2f(l)) * 0.6931471805599453f : -INFINITY;
        }
        // A thread's row sits H_q * D elements from the next one, so storing rows straight from
        // registers would touch a separate sector per lane. The rows go through this head's Q
        // buffer instead (its S MMAs have all completed, o_final being committed after them),
        // 16-byte chunks XOR-swizzled by row so both sides spread over the banks; then each warp
        // writes its own 32 rows with kChunks lanes per row. (A split launch keeps the direct
        // stores: measured, the staging slowed its key loop more than it saved.)
        if constexpr (SPLIT) {
          uint16_t *orow = p.O + (static_cast<size_t>(seq_start + row) * p.H_q + h) * D;
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tg::tmem_ld_32x32b_x32(lane_addr + colO + c0, o);
            tg::tmem_ld_wait();
            if (row < seq_len) {
              uint32_t w[16];
#pragma unroll
              for (int i = 0; i < 16; ++i)
                w[i] = tg::pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
              uint4 *dst = reinterpret_cast<uint4 *>(orow + c0);
#pragma unroll
              for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
            }
          }
        } else {
          constexpr int kChunks = D / 8;  // 16-byte chunks per row
          uint4 *stg = reinterpret_cast<uint4 *>(sQ + t * C::kTileBytes);
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tg::tmem_ld_32x32b_x32(lane_addr + colO + c0, o);
            tg::tmem_ld_wait();
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              w[i] = tg::pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              stg[r * kChunks + ((c0 / 8 + i) ^ (r & (kChunks - 1)))] =
                  make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
          }
          __syncwarp();
          constexpr int kRowsPerStep = 32 / kChunks;
          const int cl = lane % kChunks;
#pragma unroll 8
          for (int rr = 0; rr < 32; rr += kRowsPerStep) {
            const int rt = wq * 32 + rr + lane / kChunks;  // row within the tile
            const uint4 v = stg[rt * kChunks + (cl ^ (rt & (kChunks - 1)))];
            if (q0 + rt < seq_len)
              reinterpret_cast<uint4 *>(p.O + (static_cast<size_t>(seq_start + q0 + rt) * p.H_q + h) * D)[cl] = v;
          }
        }
      }
      if (!ok) *vabort = 1;
    }
    if (SPLIT && n_chunks > 1) {
      // ---- split key range: arrive; the last chunk of this query tile combines every slot ----
      // All eight warps take part (warps of an absent second head included), so the named
      // barrier always completes. A chunk that gave up still arrives, so the counter stays
      // consistent; the status word then carries TG_DEV_TIMEOUT.
      // The barrier orders every thread's partial stores before thread 128's release; its
      // acq_rel add then publishes them device-wide with the arrival, and, for the last chunk,
      // acquires every other chunk's published partial before the barrier below.
      named_bar_sync(1, 256);
      int32_t *s_last = abort_flag + 4;
      if (threadIdx.x == 128) {
        int32_t *cnt = p.ws_count + (static_cast<size_t>(b) * p.pairs + hp) * p.n_qt_max + tq;
        int prev;
        asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;" : "=r"(prev) : "l"(cnt) : "memory");
        const int last = prev == n_chunks - 1;
        if (last) *cnt = 0;  // ready for the next call on this workspace
        *s_last = last;
      }
      named_bar_sync(1, 256);
      const int row = q0 + r;
      // warp-uniform condition: the tensor-memory loads below are warp-collective
      if (*s_last && t < n_tiles) {
        const bool valid = row < seq_len;
        const int h = h0 + t;
        const uint32_t colO = t == 0 ? C::kColO0 : C::kColO1;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const float *slot0 = p.ws_part + (static_cast<size_t>(b * p.pairs + hp) * p.n_u +
                                          chunk_slot_base(tq, p.chunk)) * slot_floats<D>();
        const size_t ml_off = static_cast<size_t>(2) * 128 * D + (t * 128 + r) * 2;
        const size_t o_off = static_cast<size_t>(t) * (D / 4) * 128 + r;  // in float4, then + c4 * 128
        // This CTA's own chunk is read back from tensor memory and registers (the same values it
        // stored). The other chunks' rows sit in L2, about a thousand cycles away, so each thread
        // stages its own rows of them into the (now idle) operand buffers with asynchronous
        // 16-byte copies, 32 columns per round and up to three rounds in flight (64 KB each, in
        // the 192 KB of Q/K/V buffers; both rounds of d_h = 64 fit its 128 KB), and reads them back
        // from shared memory: about one round trip instead of one per load round. Weights 2^(m_c - M) over
        // the chunks with a non-empty sum; every sum runs in chunk order.
        const int tl = threadIdx.x - 128;  // 0..255
        constexpr int kRounds = D / 32;
        constexpr int kBufs = kRounds < 3 ? kRounds : 3;
        static_assert(kBufs * (kMaxChunks - 1) * 8 * 256 * 16 <= C::kOffBias, "staging fits the operand buffers");
        float4 *stage = reinterpret_cast<float4 *>(smem);  // [kBufs][kMaxChunks - 1][8][256]
        int rem[kMaxChunks - 1];
        int n_rem = 0;
#pragma unroll
        for (int c = 0; c < kMaxChunks; ++c)
          if (c < n_chunks && c != chunk_id && n_rem < kMaxChunks - 1) rem[n_rem++] = c;
        auto issue_round = [&](int c0) {
          float4 *dst = stage + ((c0 / 32) % kBufs) * (kMaxChunks - 1) * 8 * 256;
          for (int k = 0; k < n_rem; ++k) {
            const float4 *src = reinterpret_cast<const float4 *>(slot0 + rem[k] * slot_floats<D>()) + o_off + (c0 / 4) * 128;
            if (valid) {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tg::smem_u32(dst + (k * 8 + i) * 256 + tl)),
                             "l"(src + i * 128)
                             : "memory");
            }
          }
          asm volatile("cp.async.commit_group;" ::: "memory");
        };
#pragma unroll
        for (int rr = 0; rr < kBufs; ++rr) issue_round(rr * 32);
        float mc[kMaxChunks], lc[kMaxChunks];
#pragma unroll
        for (int c = 0; c < kMaxChunks; ++c) {
          float2 ml = make_float2(0.0f, 0.0f);
          if (c == chunk_id) ml = make_float2((m_ref == -INFINITY) ? 0.0f : m_ref, l);
          else if (valid && c < n_chunks) ml = __ldcg(reinterpret_cast<const float2 *>(slot0 + c * slot_floats<D>() + ml_off));
          mc[c] = ml.x;
          lc[c] = ml.y;
        }
        float M = -INFINITY;
#pragma unroll
        for (int c = 0; c < kMaxChunks; ++c)
          if (lc[c] > 0.0f) M = fmaxf(M, mc[c]);
        float w[kMaxChunks], L = 0.0f;
#pragma unroll
        for (int c = 0; c < kMaxChunks; ++c) {
          w[c] = lc[c] > 0.0f ? ex2(mc[c] - M) : 0.0f;
          L = fmaf(w[c], lc[c], L);
        }
        const float inv_L = L > 0.0f ? 1.0f / L : 0.0f;
        if (p.lse != nullptr && valid)
          p.lse[static_cast<size_t>(seq_start + row) * p.H_q + h] =
              L > 0.0f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
        uint16_t *orow = p.O + (static_cast<size_t>(seq_start + row) * p.H_q + h) * D;
        for (int c0 = 0; c0 < D; c0 += 32) {
          // round r has landed once at most the rounds issued after it are still in flight
          const int pending = min(kBufs - 1, kRounds - 1 - c0 / 32);
          if (pending >= 2) asm volatile("cp.async.wait_group 2;" ::: "memory");
          else if (pending == 1) asm volatile("cp.async.wait_group 1;" ::: "memory");
          else asm volatile("cp.async.wait_group 0;" ::: "memory");
          const float4 *src = stage + ((c0 / 32) % kBufs) * (kMaxChunks - 1) * 8 * 256;
          uint32_t own[32];
          tg::tmem_ld_32x32b_x32(lane_addr + colO + c0, own);
          tg::tmem_ld_wait();
          float acc[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[i] = 0.0f;
          int k = 0;
#pragma unroll
          for (int c = 0; c < kMaxChunks; ++c) {
            if (c >= n_chunks) break;
            if (c == chunk_id) {
#pragma unroll
              for (int i = 0; i < 32; ++i) acc[i] = fmaf(w[c], __uint_as_float(own[i]), acc[i]);
            } else {
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float4 x = src[(k * 8 + i) * 256 + tl];
                acc[4 * i] = fmaf(w[c], x.x, acc[4 * i]);
                acc[4 * i + 1] = fmaf(w[c], x.y, acc[4 * i + 1]);
                acc[4 * i + 2] = fmaf(w[c], x.z, acc[4 * i + 2]);
                acc[4 * i + 3] = fmaf(w[c], x.w, acc[4 * i + 3]);
              }
              ++k;
            }
          }
          if (valid) {
            uint32_t wv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) wv[i] = tg::pack_bf16x2(acc[2 * i] * inv_L, acc[2 * i + 1] * inv_L);
            uint4 *dst = reinterpret_cast<uint4 *>(orow + c0);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(wv[4 * i], wv[4 * i + 1], wv[4 * i + 2], wv[4 * i + 3]);
          }
          // this round's buffer is refilled by round r + kBufs
          if (c0 + 32 * kBufs < D) issue_round(c0 + 32 * kBufs);
        }
      }
    }
  }

  tg::tc_fence_before();
  __syncthreads();
  if (*vabort) {
    if (threadIdx.x == 0) {
      tg::report(p.status, TG_DEV_TIMEOUT);
      volatile int32_t never = 0;
      for (int i = *n_consumed; i < *n_issued; ++i)
        tg::mbar_wait(&kv_full[i % C::kStages], (i / C::kStages) & 1, &never, p.drain_limit);
      if (*q_issued) tg::mbar_wait(q_full, 0, &never, p.drain_limit);
    }
    __syncthreads();
  }
  if (warp == 1) {
    tg::tc_fence_after();
    tg::tmem_dealloc(tmem, 512);
  }
}

template <int D, int MODE>
tg_status launch_attention_d(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                             AttnParams &p, cudaStream_t stream) {
  using C = AttnCfg<D>;
  CUtensorMap tm_q, tm_k, tm_v;
  const uint32_t box[3] = {64, 1, 128};
  {
    const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(p.H_q),
                              static_cast<uint64_t>(p.M_cap)};
    const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2,
                                 static_cast<uint64_t>(p.H_q) * D * 2};
    if (!tg_host::encode_tmap_bf16(&tm_q, Q, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return TG_ERR_CUDA;
  }
  {
    const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(p.H_kv),
                              static_cast<uint64_t>(p.M_cap)};
    const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2,
                                 static_cast<uint64_t>(p.H_kv) * D * 2};
    if (!tg_host::encode_tmap_bf16(&tm_k, K, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return TG_ERR_CUDA;
    if (!tg_host::encode_tmap_bf16(&tm_v, V, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return TG_ERR_CUDA;
  }
  // a split launch is its own instantiation, so the key loop of the one-CTA-per-tile kernel keeps
  // its register allocation
  auto kernel = gated_attention_kernel<D, MODE, false>;
  if constexpr (MODE == kLogGate) {
    if (p.split) kernel = gated_attention_kernel<D, MODE, true>;
  } else {
    if (p.split) return TG_ERR_UNSUPPORTED;
  }
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return tg_host::record_cuda(e);
  const long long grid = static_cast<long long>(p.split ? p.n_u : p.n_qt_max) * p.B * p.pairs;
  if (grid == 0) return TG_OK;
  if (grid > 0x7FFFFFFFLL) return TG_ERR_UNSUPPORTED;
  return tg_host::record_cuda(tg_host::launch_pdl(kernel, dim3(static_cast<int>(grid)), dim3(kThreads),
                                                  C::kSmemBytes, stream, tm_q, tm_k, tm_v, p));
}

}  // namespace

// The split workspace of tg_gated_attention_noalloc: a fixed 16 MiB array in device memory, which
// every GPU that loads this library holds until the process exits. Host code only names it to
// look up its device address (cudaGetSymbolAddress); the kernels receive that address.
constexpr size_t kFixedScratchBytes = static_cast<size_t>(16) << 20;
static __device__ __align__(256) uint8_t g_fixed_scratch[kFixedScratchBytes];

namespace tg_host {

namespace {

// How a launch splits its key ranges (see AttnParams): only when one CTA per query tile would
// leave SMs idle. The chunk is the smallest number of key tiles for which every (query tile,
// chunk) CTA still fits in one wave on this device, so the longest CTA is as short as it can be
// without a second wave.
struct SplitPlan {
  int32_t split = 0, chunk = 0, n_u = 0;
  uint32_t tab[kMaxChunkItems] = {};
  size_t ws_bytes = 0;
};

size_t count_bytes(int32_t B, int32_t pairs, int32_t n_qt) {
  const size_t n = static_cast<size_t>(B) * pairs * n_qt * sizeof(int32_t);
  return (n + 255) & ~static_cast<size_t>(255);
}

SplitPlan plan_split(int32_t B, int32_t max_seqlen, int32_t H_q, int32_t H_kv, int32_t d_h, int sms) {
  SplitPlan sp;
  const int32_t group = H_q / H_kv;
  const int32_t pairs = H_q / ((group % 2 == 0) ? 2 : 1);
  const int32_t n_qt = (max_seqlen + kBlockM - 1) / kBlockM;
  const long long base = static_cast<long long>(n_qt) * B * pairs;
  if (n_qt < kMinSplitSteps || base >= sms) return sp;
  // at most kMaxChunks chunks per query tile: the combine keeps one register set per chunk
  for (int32_t chunk = (n_qt + kMaxChunks - 1) / kMaxChunks; chunk < n_qt; ++chunk) {
    const int32_t n_u = chunk_slot_base(n_qt, chunk);
    if (n_u > kMaxChunkItems) continue;
    if (static_cast<long long>(n_u) * B * pairs > sms) continue;
    sp.split = 1;
    sp.chunk = chunk;
    sp.n_u = n_u;
    // heaviest first: by chunk length, then by query tile (later tiles see more keys)
    int k = 0;
    for (int32_t len = chunk; len >= 1; --len)
      for (int32_t tq = n_qt - 1; tq >= 0; --tq)
        for (int32_t c = 0; c * chunk <= tq; ++c)
          if (std::min(chunk, tq + 1 - c * chunk) == len) sp.tab[k++] = static_cast<uint32_t>(tq) | (static_cast<uint32_t>(c) << 16);
    const size_t slot = d_h == 128 ? slot_floats<128>() : slot_floats<64>();
    sp.ws_bytes = count_bytes(B, pairs, n_qt) + static_cast<size_t>(B) * pairs * n_u * slot * sizeof(float);
    return sp;
  }
  return sp;
}

AttnParams common_params(const float *bias_src, int32_t H_g, const int32_t *pos, const int32_t *cu_kept,
                         int32_t B, int32_t M_cap, int32_t max_seqlen, int32_t H_q, int32_t H_kv, uint16_t *O,
                         int32_t *status) {
  AttnParams p;
  p.lse = nullptr;
  p.g = bias_src;
  p.g_cols = H_g;
  p.g_group = H_q / H_g;
  p.pos = pos;
  p.cu_kept = cu_kept;
  p.B = B;
  p.M_cap = M_cap;
  p.max_seqlen = max_seqlen;
  p.H_q = H_q;
  p.H_kv = H_kv;
  p.group = H_q / H_kv;
  p.heads_per_cta = (p.group % 2 == 0) ? 2 : 1;
  p.pairs = H_q / p.heads_per_cta;
  p.n_qt_max = (max_seqlen + kBlockM - 1) / kBlockM;
  p.O = O;
  p.status = status;
  p.wait_limit = wait_limit_ns();
  p.drain_limit = drain_limit_ns();
  p.withhold = (withhold_mask() & TG_WITHHOLD_ATTENTION) != 0;
  p.split = 0;
  p.chunk = 0;
  p.n_u = 0;
  p.ws_count = nullptr;
  p.ws_part = nullptr;
  return p;
}

// Take the split plan when a workspace is given; a split launch needs plan.ws_bytes of it.
tg_status apply_split(AttnParams &p, int32_t d_h, void *workspace, size_t workspace_bytes) {
  if (workspace == nullptr) return TG_OK;
  const SplitPlan sp = plan_split(p.B, p.max_seqlen, p.H_q, p.H_kv, d_h, num_sms());
  if (!sp.split) return TG_OK;
  if (workspace_bytes < sp.ws_bytes) return TG_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return TG_ERR_INVALID_ARG;
  p.split = 1;
  p.chunk = sp.chunk;
  p.n_u = sp.n_u;
  for (int i = 0; i < kMaxChunkItems; ++i) p.u_tab[i] = sp.tab[i];
  p.ws_count = static_cast<int32_t *>(workspace);
  p.ws_part = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + count_bytes(p.B, p.pairs, p.n_qt_max));
  return TG_OK;
}

}  // namespace

size_t gated_attention_workspace_size(int32_t B, int32_t max_seqlen, int32_t H_q, int32_t H_kv, int32_t d_h) {
  if (B < 1 || max_seqlen < 1 || H_q < 1 || H_kv < 1 || H_q % H_kv != 0 || (d_h != 64 && d_h != 128)) return 0;
  return plan_split(B, max_seqlen, H_q, H_kv, d_h, num_sms()).ws_bytes;
}

tg_status launch_gated_attention(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                                 const float *g, int32_t H_g, const int32_t *cu_kept, int32_t B,
                                 int32_t M_cap, int32_t max_seqlen, int32_t H_q, int32_t H_kv,
                                 int32_t d_h, const float *tau, const float *beta, uint16_t *O,
                                 int32_t *status, cudaStream_t stream, float *lse, void *workspace,
                                 size_t workspace_bytes) {
  if (M_cap == 0 || max_seqlen == 0) return TG_OK;
  AttnParams p = common_params(g, H_g, nullptr, cu_kept, B, M_cap, max_seqlen, H_q, H_kv, O, status);
  p.lse = lse;
  const tg_status st = apply_split(p, d_h, workspace, workspace_bytes);
  if (st != TG_OK) return st;
  const float log2e = 1.4426950408889634f;
  for (int h = 0; h < kMaxHeads; ++h) {
    p.scale_log2[h] = h < H_q ? tau[h] * log2e / std::sqrt(static_cast<float>(d_h)) : 0.0f;
    p.beta[h] = h < H_q ? beta[h] : 0.0f;
  }
  if (d_h == 128) return launch_attention_d<128, kLogGate>(Q, K, V, p, stream);
  if (d_h == 64) return launch_attention_d<64, kLogGate>(Q, K, V, p, stream);
  return TG_ERR_UNSUPPORTED;
}

tg_status launch_gated_attention_eq8(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                                     const float *b, int32_t H_g, const int32_t *pos, const int32_t *cu_kept,
                                     int32_t B, int32_t M_cap, int32_t max_seqlen, int32_t H_q,
                                     int32_t H_kv, int32_t d_h, const float *gain,
                                     const float *temp, uint16_t *O, int32_t *status,
                                     cudaStream_t stream) {
  if (M_cap == 0 || max_seqlen == 0) return TG_OK;
  AttnParams p = common_params(b, H_g, pos, cu_kept, B, M_cap, max_seqlen, H_q, H_kv, O, status);
  const float log2e = 1.4426950408889634f;
  for (int h = 0; h < kMaxHeads; ++h) {
    p.scale_log2[h] = h < H_q ? temp[h] : 0.0f;
    p.beta[h] = h < H_q ? gain[h] * log2e : 0.0f;
  }
  if (d_h == 128) return launch_attention_d<128, kEq8>(Q, K, V, p, stream);
  if (d_h == 64) return launch_attention_d<64, kEq8>(Q, K, V, p, stream);
  return TG_ERR_UNSUPPORTED;
}

// ---------------------------------------------------------------------------
// Attention for callers that cannot allocate device memory (tg_gated_attention_noalloc): the
// split launch's workspace is a fixed array that the library itself holds on the device, so
// such a caller never needs to hand one in. Its address is looked up once per device.
// ---------------------------------------------------------------------------

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_fixed_scratch_mu;
void *g_fixed_scratch_ptr[kMaxDevices] = {};

// Device address of the fixed scratch array on the current device (looked up on first use).
tg_status fixed_scratch(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return record_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return TG_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_fixed_scratch_mu);
  if (g_fixed_scratch_ptr[dev] == nullptr) {
    void *ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_fixed_scratch);
    if (e != cudaSuccess) return record_cuda(e);
    g_fixed_scratch_ptr[dev] = ptr;
  }
  *out = g_fixed_scratch_ptr[dev];
  return TG_OK;
}

}  // namespace

tg_status launch_gated_attention_noalloc(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                                         const float *g, int32_t H_g, const int32_t *cu_kept, int32_t B,
                                         int32_t M_cap, int32_t max_seqlen, int32_t H_q, int32_t H_kv,
                                         int32_t d_h, const float *tau, const float *beta, uint16_t *O,
                                         int32_t *status, cudaStream_t stream) {
  if (M_cap == 0 || max_seqlen == 0) return TG_OK;
  const size_t need = gated_attention_workspace_size(B, max_seqlen, H_q, H_kv, d_h);
  if (need > kFixedScratchBytes) return TG_ERR_UNSUPPORTED;  // more than the fixed array holds
  void *scratch = nullptr;
  if (need > 0) {
    const tg_status st = fixed_scratch(&scratch);
    if (st != TG_OK) return st;
    // the array keeps the previous call's contents: its arrival counters must start at zero
    const int32_t pairs = H_q / (((H_q / H_kv) % 2 == 0) ? 2 : 1);
    const cudaError_t e =
        cudaMemsetAsync(scratch, 0, count_bytes(B, pairs, (max_seqlen + kBlockM - 1) / kBlockM), stream);
    if (e != cudaSuccess) return record_cuda(e);
  }
  return launch_gated_attention(Q, K, V, g, H_g, cu_kept, B, M_cap, max_seqlen, H_q, H_kv, d_h, tau, beta, O,
                                status, stream, nullptr, scratch, need > 0 ? kFixedScratchBytes : 0);
}

}  // namespace tg_host
