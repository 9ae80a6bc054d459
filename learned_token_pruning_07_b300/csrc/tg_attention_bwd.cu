// tg_attention_bwd.cu — backward of token-gated attention (TokenGate deep dive, section 3.2:
// the gate score reaches the loss only through the per-key attention bias, Eq. (5)/(8); the
// top-K choice itself carries no gradient, section 3.1), and the gate-score gradient.
//
// For one sequence and query head h (kv head h / group), with x_ij = c_h q_i.k_j + beta_h ln g_j
// over j <= i (c_h = tau_h / sqrt(d_h)) and P_ij = exp(x_ij - LSE_i) (LSE from the forward):
//   dP_ij = dO_i . v_j,  D_i = dO_i . o_i,  dX_ij = P_ij (dP_ij - D_i)
//   dV_j = sum_i P_ij dO_i,  dK_j = c_h sum_i dX_ij q_i,
//   dQ_i = c_h sum_j dX_ij k_j,  dbias_jh = sum_i dX_ij.
//
// Three launches, all on the tensor cores except the first:
//   1. bwd_rowdot_kernel: D_i = dO_i . o_i per kept row and query head (fp32 sums of the bf16
//      values). It is parked in the first element of that row's dQ, which nothing else uses
//      until pass 3 writes dQ, so the backward needs no scratch memory.
//   2. bwd_dkdv_kernel: one CTA per (128-key tile, kv head). It loops over the query heads of
//      the GQA group in head order and over the query tiles at or after its key tile:
//        S^T = K Q^T, dP^T = V dO^T (tcgen05, fp32 in tensor memory)
//        P^T, dX^T by the CUDA cores (thread = key, 128 query columns)
//        dV += P^T dO, dK += (c_h dX^T) Q (tcgen05, A operand from tensor memory, bf16)
//      dbias_jh = sum_i dX_ij is summed in fp32 by the key's thread. dK and dV stay in tensor
//      memory until the last query tile.
//   3. bwd_dq_kernel: one CTA per (128-query tile, query head). It loops over the key tiles at or
//      before its query tile: S = Q K^T, dP = dO V^T, dX as above (thread = query), and
//      dQ += (c_h dX) K.
// Both tensor-core passes are software-pipelined: the products of the next tile start as soon
// as the elementwise warps have released the tensor-memory columns they overwrite, so they
// run while the current tile's elementwise step is still working.
// Every output element is written by exactly one CTA after sums in a fixed order: the results
// are deterministic, with no atomics.
//
// Precision: the products P dO, dX q and dX k take P and c_h dX rounded to bf16 (the tensor
// cores' operand type) with fp32 accumulation; everything else is fp32.
//
// Warp roles in passes 2 and 3 (12 warps): warp 0 TMA, warp 1 tensor-memory owner and MMA issue
// (the warp runs converged, one elected lane issues), warp 2 column producer (per-column terms
// of the elementwise step), warps 4-11 the elementwise step: warps 4-7 take columns 0-63 and
// warps 8-11 columns 64-127 of the same 128 rows (warp w reads tensor-memory lanes
// 32 (w % 4) .. +31). Every wait is bounded (see tg_set_wait_limit_ns).
#include "tg_common.cuh"

namespace {

constexpr int kTile = 128;          // rows of a key or query tile
constexpr int kThreads = 384;
constexpr int kMaxHeads = 128;
constexpr float kLog2e = 1.4426950408889634f;

struct BwdParams {
  const uint16_t *O, *dO;
  const float *g;
  int32_t g_cols, g_group;  // gate heads per row (H_g); query heads per gate head
  const float *lse;
  const int32_t *cu_kept;
  int32_t B, M_cap, max_seqlen, H_q, H_kv, group, n_tiles;
  float *dQ, *dK, *dV, *dbias;
  int32_t *status;
  uint64_t wait_limit, drain_limit;
  int32_t withhold;  // test hook: the TMA warps issue no loads, so the consumers' waits run out
  float scale[kMaxHeads];  // c_h = tau_h / sqrt(d_h)
  float beta[kMaxHeads];
};

// Shared-memory layout of passes 2 and 3. Operand tiles are 128 rows of D bf16, stored by TMA as
// D / 64 halves of 128-byte-swizzled rows (16 KB per half at D = 128), as in the forward.
// Pass 2 keeps K and V for the whole CTA and streams (Q, dO) pairs; pass 3 keeps Q and dO and
// streams (K, V) pairs.
template <int D>
struct BwdCfg {
  static constexpr int kHalves = D / 64;
  static constexpr uint32_t kTileBytes = kTile * D * 2u;
  static constexpr int kStages = D == 128 ? 2 : 3;  // at D = 64 the deeper ring also keeps one CTA per SM
  static constexpr uint32_t kOffFixA = 0;                     // K (pass 2) or Q (pass 3)
  static constexpr uint32_t kOffFixB = kTileBytes;            // V (pass 2) or dO (pass 3)
  static constexpr uint32_t kOffRing = 2 * kTileBytes;        // [stage] { Q | K, dO | V }
  static constexpr uint32_t kOffCols = kOffRing + kStages * 2 * kTileBytes;  // [2 slots][2][128] f32
  static constexpr uint32_t kOffXchg = kOffCols + 2 * 2 * 128 * 4;           // [128] f32
  static constexpr uint32_t kOffBar = kOffXchg + 128 * 4;
  static constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;
  // tensor memory columns: S (or S^T), dP (or dP^T), then the accumulators
  static constexpr uint32_t kColS = 0, kColDP = 128, kColAcc0 = 256, kColAcc1 = 256 + D;
  // pass 3 keeps one accumulator, so dP (and c dX in its place) alternates between kColDP and 384
  static __device__ __forceinline__ uint32_t dp_col(int j) { return (j & 1) ? 384u : kColDP; }
  static_assert(D <= 128, "pass 3's second dP block starts at column 384");
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

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

// Sequence bounds of sequence b clamped to the capacity; false (and TG_DEV_BAD_SEQLENS) when
// cu_kept is not a valid partition there.
__device__ __forceinline__ bool seq_bounds(const BwdParams &p, int b, int &start, int &len) {
  int s0 = p.cu_kept[b], s1 = p.cu_kept[b + 1];
  if (s0 < 0 || s1 < s0 || s1 - s0 > p.max_seqlen) return false;
  s0 = min(s0, p.M_cap);
  s1 = min(s1, p.M_cap);
  start = s0;
  len = s1 - s0;
  return true;
}

// ---- pass 1: D_i = dO_i . o_i, one warp per (kept row, query head), parked in dQ[i, h, 0] ----
template <int D>
__global__ void __launch_bounds__(256) bwd_rowdot_kernel(const __grid_constant__ BwdParams p) {
  tg::pdl_wait();
  tg::pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int M = max(0, min(p.cu_kept[p.B], p.M_cap));
  const long long n = static_cast<long long>(M) * p.H_q;
  const long long stride = static_cast<long long>(gridDim.x) * 8;
  for (long long w = blockIdx.x * 8LL + (threadIdx.x >> 5); w < n; w += stride) {
    const uint16_t *o = p.O + w * D, *d = p.dO + w * D;
    float acc = 0.0f;
#pragma unroll
    for (int c = lane; c < D; c += 32) acc = fmaf(tg::bf16_bits_to_float(o[c]), tg::bf16_bits_to_float(d[c]), acc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
    if (lane == 0) p.dQ[w * D] = acc;
  }
}

// All threads of named barrier `id` (count threads) arrive; returns true when `pred` held in every
// one of them. Used so that the elementwise warps leave their loop together after a wait gives
// up (a lone warp would leave the others waiting on the named barrier).
__device__ __forceinline__ bool barrier_all(uint32_t id, uint32_t count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pin, pout;\n\tsetp.ne.u32 pin, %1, 0;\n\t"
      "barrier.red.and.pred pout, %2, %3, pin;\n\tselp.u32 %0, 1, 0, pout;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void barrier_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// MMA helpers of passes 2 and 3. One 128 x 128 x D product over two K-major operand tiles
// (a K-step of 16 is 32 bytes into a 128-byte swizzled row; d-halves are 16 KB apart).
template <int D>
__device__ __forceinline__ void mma_tile_ss(uint32_t dst, uint64_t a0, uint64_t b0, uint32_t idesc) {
#pragma unroll
  for (int k = 0; k < D / 16; ++k) {
    const uint32_t off16 = ((k / 4) * 16384 + (k % 4) * 32) >> 4;
    tg::mma_bf16_ss_elect(dst, a0 + off16, b0 + off16, idesc, k != 0);
  }
}

// dst (+)= A[tensor memory, 128 rows x 128 bf16 columns] * B[128 x D, MN-major in shared memory].
// The A columns of the two 64-wide halves sit at src and src + 64 (packed bf16 pairs: 8 columns
// per 16-element K-step); B rows (the K index) step by 16 rows = 2 KB.
template <int D>
__device__ __forceinline__ void mma_tile_ts(uint32_t dst, uint32_t src, uint64_t b0, uint32_t idesc, bool first) {
#pragma unroll
  for (int k = 0; k < kTile / 16; ++k) {
    const uint32_t a = src + (k < 4 ? k * 8 : 64 + (k - 4) * 8);
    tg::mma_bf16_ts_elect(dst, a, b0 + ((k * 2048) >> 4), idesc, !(first && k == 0));
  }
}

// ---- pass 2: dK, dV and dbias for one (key tile, kv head) ----
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sK = smem + C::kOffFixA;
  uint8_t *sV = smem + C::kOffFixB;
  uint8_t *sRing = smem + C::kOffRing;            // stage s: Q at 2 s tiles, dO one tile after
  float *sCols = reinterpret_cast<float *>(smem + C::kOffCols);  // slot: [-lse_i log2 e | D_i]
  float *sX = reinterpret_cast<float *>(smem + C::kOffXchg);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
  uint64_t *kv_full = bars;
  uint64_t *ring_full = kv_full + 1;               // [kStages]
  uint64_t *ring_empty = ring_full + C::kStages;   // [kStages]
  uint64_t *s_full = ring_empty + C::kStages;      // S^T of the iteration is ready
  uint64_t *dp_full = s_full + 1;                  // dP^T of the iteration is ready
  uint64_t *p_full = dp_full + 1;                  // P^T written back (8 warps)
  uint64_t *x_full = p_full + 1;                   // c dX^T written back (8 warps)
  uint64_t *dv_done = x_full + 1;
  uint64_t *dk_done = dv_done + 1;
  uint64_t *acc_final = dk_done + 1;
  uint64_t *col_full = acc_final + 1;              // [2]
  uint64_t *col_empty = col_full + 2;              // [2]
  uint64_t *drain = col_empty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  int32_t *flags = reinterpret_cast<int32_t *>(tmem_slot + 1);  // abort, ring issued/consumed, kv issued
  volatile int32_t *vabort = flags;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  tg::pdl_wait();
  tg::pdl_launch_dependents();
  // ---- work item: key tile kt of kv head kvh in sequence b (low kt first: they have the most work) ----
  const int kvh = blockIdx.x % p.H_kv;
  const int rest = blockIdx.x / p.H_kv;
  const int b = rest % p.B;
  const int kt = rest / p.B;
  int seq_start, seq_len;
  if (!seq_bounds(p, b, seq_start, seq_len)) {
    if (threadIdx.x == 0 && kt == 0 && kvh == 0) tg::report(p.status, TG_DEV_BAD_SEQLENS);
    return;
  }
  const int k0 = kt * kTile;
  if (k0 >= seq_len) return;  // uniform for the CTA
  const int n_qt = (seq_len + kTile - 1) / kTile;
  const int n_q = n_qt - kt;          // query tiles kt .. n_qt - 1 see these keys
  const int n_iter = p.group * n_q;   // iteration i: head kvh * group + i / n_q, query tile kt + i % n_q

  if (threadIdx.x == 0) {
    tg::mbar_init(kv_full, 1);
    for (int s = 0; s < C::kStages; ++s) {
      tg::mbar_init(&ring_full[s], 1);
      tg::mbar_init(&ring_empty[s], 1);
    }
    tg::mbar_init(s_full, 1);
    tg::mbar_init(dp_full, 1);
    tg::mbar_init(p_full, 8);
    tg::mbar_init(x_full, 8);
    tg::mbar_init(dv_done, 1);
    tg::mbar_init(dk_done, 1);
    tg::mbar_init(acc_final, 1);
    for (int s = 0; s < 2; ++s) {
      tg::mbar_init(&col_full[s], 32);
      tg::mbar_init(&col_empty[s], 8);
    }
    tg::mbar_init(drain, 1);
    for (int i = 0; i < 4; ++i) flags[i] = 0;
    tg::fence_mbar_init();
    tg::prefetch_tensormap(&tm_q);
    tg::prefetch_tensormap(&tm_k);
    tg::prefetch_tensormap(&tm_v);
    tg::prefetch_tensormap(&tm_do);
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
      // ---------------- TMA: K, V of the key tile once; then (Q, dO) of every iteration ----------------
      tg::mbar_arrive_expect_tx(kv_full, 2 * C::kTileBytes);
      for (int hf = 0; hf < C::kHalves; ++hf) {
        tg::tma_load_3d(sK + hf * 16384, &tm_k, kv_full, hf * 64, kvh, seq_start + k0);
        tg::tma_load_3d(sV + hf * 16384, &tm_v, kv_full, hf * 64, kvh, seq_start + k0);
      }
      flags[3] = 1;
      for (int i = 0; i < n_iter; ++i) {
        const int s = i % C::kStages;
        const int h = kvh * p.group + i / n_q, q0 = (kt + i % n_q) * kTile;
        if (!tg::mbar_wait(&ring_empty[s], ((i / C::kStages) & 1) ^ 1u, vabort, p.wait_limit)) {
          *vabort = 1;
          break;
        }
        uint8_t *dst = sRing + s * 2 * C::kTileBytes;
        tg::mbar_arrive_expect_tx(&ring_full[s], 2 * C::kTileBytes);
        for (int hf = 0; hf < C::kHalves; ++hf) {
          tg::tma_load_3d(dst + hf * 16384, &tm_q, &ring_full[s], hf * 64, h, seq_start + q0);
          tg::tma_load_3d(dst + C::kTileBytes + hf * 16384, &tm_do, &ring_full[s], hf * 64, h, seq_start + q0);
        }
        flags[1] = i + 1;
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issue (converged warp, elected lane) ----------------
    // Software-pipelined: dV(i) starts once P^T(i) is written, S^T(i + 1) refills those columns once
    // dV(i) has read them, and dK(i) then dP^T(i + 1) follow c dX^T(i) in the same way, so the
    // products of one iteration run while the elementwise warps work on the other half of it.
    const uint32_t idesc_st = tg::idesc_bf16_f32(kTile, kTile);          // K Q^T, V dO^T: both K-major
    const uint32_t idesc_acc = tg::idesc_bf16_f32(kTile, D, 0, 1);       // P^T dO, dX^T Q: B MN-major
    const uint64_t dk0 = tg::smem_desc(tg::smem_u32(sK), 16, 1024, tg::kSwz128);
    const uint64_t dv0 = tg::smem_desc(tg::smem_u32(sV), 16, 1024, tg::kSwz128);
    const uint64_t dr0 = tg::smem_desc(tg::smem_u32(sRing), 16, 1024, tg::kSwz128);
    const uint64_t dr0_mn = tg::smem_desc(tg::smem_u32(sRing), 16384, 1024, tg::kSwz128);
    constexpr uint32_t kTile16 = C::kTileBytes >> 4;
    bool ok = __all_sync(0xFFFFFFFFu, tg::mbar_wait(kv_full, 0, vabort, p.wait_limit));
    if (ok) ok = __all_sync(0xFFFFFFFFu, tg::mbar_wait(&ring_full[0], 0, vabort, p.wait_limit));
    int consumed = 0;
    if (ok) {  // S^T(0), dP^T(0): ring stage 0 holds Q at tile 0, dO at tile 1
      consumed = 1;
      tg::tc_fence_after();
      mma_tile_ss<D>(tmem + C::kColS, dk0, dr0, idesc_st);
      tg::mma_commit_elect(s_full);
      mma_tile_ss<D>(tmem + C::kColDP, dv0, dr0 + kTile16, idesc_st);
      tg::mma_commit_elect(dp_full);
    }
    for (int i = 0; i < n_iter && ok; ++i) {
      const int s = i % C::kStages, s1 = (i + 1) % C::kStages;
      const uint64_t q_off = 2 * s * kTile16, do_off = q_off + kTile16;
      const uint64_t q1_off = 2 * s1 * kTile16, do1_off = q1_off + kTile16;
      const bool more = i + 1 < n_iter;
      ok = __all_sync(0xFFFFFFFFu, tg::mbar_wait(p_full, i & 1, vabort, p.wait_limit));
      if (!ok) break;
      tg::tc_fence_after();
      mma_tile_ts<D>(tmem + C::kColAcc0, tmem + C::kColS, dr0_mn + do_off, idesc_acc, i == 0);   // dV
      tg::mma_commit_elect(dv_done);
      if (more) {  // S^T(i + 1) overwrites P^T(i): after dV(i) has read it
        ok = __all_sync(0xFFFFFFFFu, tg::mbar_wait(&ring_full[s1], ((i + 1) / C::kStages) & 1, vabort,
                                                   p.wait_limit));
        if (ok) ok = __all_sync(0xFFFFFFFFu, tg::mbar_wait(dv_done, i & 1, vabort, p.wait_limit));
        if (!ok) break;
        consumed = i + 2;
        tg::tc_fence_after();
        mma_tile_ss<D>(tmem + C::kColS, dk0, dr0 + q1_off, idesc_st);
        tg::mma_commit_elect(s_full);
      }
      ok = __all_sync(0xFFFFFFFFu, tg::mbar_wait(x_full, i & 1, vabort, p.wait_limit));
      if (!ok) break;
      tg::tc_fence_after();
      mma_tile_ts<D>(tmem + C::kColAcc1, tmem + C::kColDP, dr0_mn + q_off, idesc_acc, i == 0);   // dK
      tg::mma_commit_elect(dk_done);
      tg::mma_commit_elect(&ring_empty[s]);
      if (more) {  // dP^T(i + 1) overwrites c dX^T(i): after dK(i) has read it
        ok = __all_sync(0xFFFFFFFFu, tg::mbar_wait(dk_done, i & 1, vabort, p.wait_limit));
        if (!ok) break;
        tg::tc_fence_after();
        mma_tile_ss<D>(tmem + C::kColDP, dv0, dr0 + do1_off, idesc_st);
        tg::mma_commit_elect(dp_full);
      }
    }
    if (ok) tg::mma_commit_elect(acc_final);
    if (lane == 0) flags[2] = consumed;
    if (!ok) {
      *vabort = 1;
      tg::mma_commit_elect(drain);
      volatile int32_t never = 0;
      tg::mbar_wait(drain, 0, &never, p.drain_limit);
    }
  } else if (warp == 2) {
    // ---------------- column producer: -LSE_i log2 e and D_i of the iteration's 128 queries ----------------
    // Queries past the sequence (or with no visible weight, LSE = -inf) get -inf, so their P is 0.
    for (int i = 0; i < n_iter; ++i) {
      const int slot = i & 1;
      const int h = kvh * p.group + i / n_q, q0 = (kt + i % n_q) * kTile;
      if (!tg::mbar_wait(&col_empty[slot], ((i >> 1) & 1) ^ 1u, vabort, p.wait_limit)) {
        *vabort = 1;
        break;
      }
      float *dst = sCols + slot * 256;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int q = lane * 4 + u, qi = q0 + q;
        float negl = -INFINITY, dd = 0.0f;
        if (qi < seq_len) {
          const size_t row = static_cast<size_t>(seq_start + qi) * p.H_q + h;
          const float lse = p.lse[row];
          if (lse > -INFINITY) negl = -lse * kLog2e;
          dd = p.dQ[row * D];
        }
        dst[q] = negl;
        dst[128 + q] = -dd;  // -D_i: the elementwise step adds it
      }
      tg::mbar_arrive(&col_full[slot]);
    }
  } else if (warp >= 4) {
    // ---------------- elementwise: thread = key row, warps 4-7 / 8-11 = query columns 0-63 / 64-127 ----------------
    // Two halves per iteration: P^T from S^T (signals p_full, so dV starts), then c dX^T from dP^T with
    // P kept in registers (signals x_full, so dK starts).
    const int wq = warp & 3, hh = (warp - 4) >> 2;
    const int k = wq * 32 + lane, kj = k0 + k;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    float dbias_acc = 0.0f, bias2 = 0.0f, c2 = 0.0f, ch = 0.0f;
    bool ok = true;
    for (int i = 0; i < n_iter; ++i) {
      const int gi = i / n_q, qt = kt + i % n_q, h = kvh * p.group + gi, slot = i & 1;
      if (i % n_q == 0) {
        // a new query head: this key's bias beta_h log2 g_j and the logit scale
        bias2 = 0.0f;
        if (p.g != nullptr && p.beta[h] != 0.0f && kj < seq_len) {
          const float lg = tg::log2_gate(p.g[static_cast<size_t>(seq_start + kj) * p.g_cols + h / p.g_group]);
          bias2 = p.beta[h] * lg;
        }
        ch = p.scale[h];
        c2 = ch * kLog2e;
      }
      bool w = tg::mbar_wait(s_full, i & 1, vabort, p.wait_limit);
      w = w && tg::mbar_wait(&col_full[slot], (i >> 1) & 1, vabort, p.wait_limit);
      ok = barrier_all(1, 256, w);  // the same decision in all eight warps
      if (!ok) break;
      tg::tc_fence_after();
      const float *negl = sCols + slot * 256, *negd = negl + 128;
      const bool diag = qt == kt;
      const uint64_t c2x = f2(c2, c2), chx = f2(ch, ch), b2x = f2(bias2, bias2);
      // ---- first half: P^T ----
      uint32_t pv[2][32];
      tg::tmem_ld_32x32b_x32(lane_addr + C::kColS + 64 * hh, pv[0]);
      tg::tmem_ld_32x32b_x32(lane_addr + C::kColS + 64 * hh + 32, pv[1]);
      tg::tmem_ld_wait();
#pragma unroll
      for (int chunk = 0; chunk < 2; ++chunk) {
        const int c0 = 64 * hh + 32 * chunk;
        uint32_t *sv = pv[chunk];
        const float4 *nl4 = reinterpret_cast<const float4 *>(negl + c0);
        // the 32 logits in log2 units, in place
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 nl = nl4[c4];
          const uint64_t a = f2_fma(f2(__uint_as_float(sv[4 * c4]), __uint_as_float(sv[4 * c4 + 1])), c2x,
                                    f2_add(b2x, f2(nl.x, nl.y)));
          const uint64_t b = f2_fma(f2(__uint_as_float(sv[4 * c4 + 2]), __uint_as_float(sv[4 * c4 + 3])), c2x,
                                    f2_add(b2x, f2(nl.z, nl.w)));
          float a0, a1, b0, b1;
          f2_split(a, a0, a1);
          f2_split(b, b0, b1);
          sv[4 * c4] = __float_as_uint(a0);
          sv[4 * c4 + 1] = __float_as_uint(a1);
          sv[4 * c4 + 2] = __float_as_uint(b0);
          sv[4 * c4 + 3] = __float_as_uint(b1);
        }
        // the 32 exponentials back to back
#pragma unroll
        for (int c = 0; c < 32; ++c) sv[c] = __float_as_uint(ex2(__uint_as_float(sv[c])));
        if (diag) {  // query before key: not visible
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (c0 + c < k) sv[c] = 0u;
        }
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) pk[c / 2] = tg::pack_bf16x2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1]));
        tg::tmem_st_32x32b_x16(lane_addr + C::kColS + 64 * hh + 16 * chunk, pk);
      }
      tg::tmem_st_wait();
      tg::tc_fence_before();
      __syncwarp();
      if (lane == 0) tg::mbar_arrive(p_full);
      // ---- second half: c dX^T = c P (dP - D), and the bias gradient ----
      w = tg::mbar_wait(dp_full, i & 1, vabort, p.wait_limit);
      ok = barrier_all(1, 256, w);
      if (!ok) break;
      tg::tc_fence_after();
      uint64_t db2[2] = {f2(0.0f, 0.0f), f2(0.0f, 0.0f)};
#pragma unroll
      for (int chunk = 0; chunk < 2; ++chunk) {
        const int c0 = 64 * hh + 32 * chunk;
        const uint32_t *sv = pv[chunk];
        uint32_t dpv[32], xk[16];
        tg::tmem_ld_32x32b_x32(lane_addr + C::kColDP + c0, dpv);
        tg::tmem_ld_wait();
        const float4 *nd4 = reinterpret_cast<const float4 *>(negd + c0);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 nd = nd4[c4];
          const float ndv[4] = {nd.x, nd.y, nd.z, nd.w};
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int c = 4 * c4 + 2 * u;
            const uint64_t xx = f2_mul(f2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])),
                                       f2_add(f2(__uint_as_float(dpv[c]), __uint_as_float(dpv[c + 1])),
                                              f2(ndv[2 * u], ndv[2 * u + 1])));
            db2[u] = f2_add(db2[u], xx);
            float s0, s1;
            f2_split(f2_mul(xx, chx), s0, s1);
            xk[c / 2] = tg::pack_bf16x2(s0, s1);
          }
        }
        tg::tmem_st_32x32b_x16(lane_addr + C::kColDP + 64 * hh + 16 * chunk, xk);
      }
      {
        float a0, a1, b0, b1;
        f2_split(db2[0], a0, a1);
        f2_split(db2[1], b0, b1);
        dbias_acc += (a0 + a1) + (b0 + b1);
      }
      tg::tmem_st_wait();
      tg::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        tg::mbar_arrive(x_full);
        tg::mbar_arrive(&col_empty[slot]);
      }
      if (i % n_q == n_q - 1) {
        // last query tile of head h: dbias_jh = half 0 + half 1
        if (hh == 1) sX[k] = dbias_acc;
        barrier_sync(1, 256);
        if (hh == 0 && kj < seq_len) p.dbias[static_cast<size_t>(seq_start + kj) * p.H_q + h] = dbias_acc + sX[k];
        barrier_sync(1, 256);
        dbias_acc = 0.0f;
      }
    }
    // ---- epilogue: dV (warps 4-7) and dK (warps 8-11) rows of this key tile ----
    if (ok) ok = __all_sync(0xFFFFFFFFu, tg::mbar_wait(acc_final, 0, vabort, p.wait_limit));
    if (ok) {
      tg::tc_fence_after();
      // Rows sit H_kv * D floats apart, so a thread storing its own row would touch a separate
      // sector per lane. The rows go through shared memory instead (K, V and the ring are idle once
      // acc_final has fired: dV in the K and V buffers, dK in the ring), 16-byte chunks
      // XOR-swizzled by row, and each warp then writes its own 32 rows with kCh lanes per row.
      constexpr int kCh = D / 4;  // 16-byte chunks per fp32 row
      float4 *stg = reinterpret_cast<float4 *>(hh == 0 ? smem + C::kOffFixA : sRing);
      const uint32_t col = hh == 0 ? C::kColAcc0 : C::kColAcc1;
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t v[32];
        tg::tmem_ld_32x32b_x32(lane_addr + col + c0, v);
        tg::tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 8; ++u)
          stg[k * kCh + ((c0 / 4 + u) ^ (k & (kCh - 1)))] =
              make_float4(__uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]), __uint_as_float(v[4 * u + 2]),
                          __uint_as_float(v[4 * u + 3]));
      }
      __syncwarp();
      float *out0 = hh == 0 ? p.dV : p.dK;
      const int cl = lane % kCh;
#pragma unroll 8
      for (int rr = 0; rr < 32; rr += 32 / kCh) {
        const int kt = wq * 32 + rr + lane / kCh;  // key row within the tile
        const float4 v = stg[kt * kCh + (cl ^ (kt & (kCh - 1)))];
        if (k0 + kt < seq_len)
          reinterpret_cast<float4 *>(out0 + (static_cast<size_t>(seq_start + k0 + kt) * p.H_kv + kvh) * D)[cl] = v;
      }
    } else {
      *vabort = 1;
    }
  }

  tg::tc_fence_before();
  __syncthreads();
  if (*vabort) {
    if (threadIdx.x == 0) {
      tg::report(p.status, TG_DEV_TIMEOUT);
      volatile int32_t never = 0;
      for (int i = flags[2]; i < flags[1]; ++i)
        tg::mbar_wait(&ring_full[i % C::kStages], (i / C::kStages) & 1, &never, p.drain_limit);
      if (flags[3]) tg::mbar_wait(kv_full, 0, &never, p.drain_limit);
    }
    __syncthreads();
  }
  if (warp == 1) {
    tg::tc_fence_after();
    tg::tmem_dealloc(tmem, 512);
  }
}

// ---- pass 3: dQ for one (query tile, query head) ----
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = smem + C::kOffFixA;
  uint8_t *sdO = smem + C::kOffFixB;
  uint8_t *sRing = smem + C::kOffRing;            // stage s: K at 2 s tiles, V one tile after
  float *sCols = reinterpret_cast<float *>(smem + C::kOffCols);  // slot: beta_h log2 g_j of 128 keys
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
  uint64_t *qd_full = bars;
  uint64_t *ring_full = qd_full + 1;               // [kStages]
  uint64_t *ring_empty = ring_full + C::kStages;   // [kStages]
  uint64_t *st_full = ring_empty + C::kStages;     // S and dP of the iteration are ready
  uint64_t *s_free = st_full + 1;                  // S read into registers (8 warps)
  uint64_t *p_full = s_free + 1;                   // [2] c dX of iteration j written back (8 warps)
  uint64_t *dq_done = p_full + 2;
  uint64_t *acc_final = dq_done + 1;
  uint64_t *col_full = acc_final + 1;              // [2]
  uint64_t *col_empty = col_full + 2;              // [2]
  uint64_t *drain = col_empty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  int32_t *flags = reinterpret_cast<int32_t *>(tmem_slot + 1);  // abort, ring issued/consumed, q issued
  volatile int32_t *vabort = flags;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  tg::pdl_wait();
  tg::pdl_launch_dependents();
  // ---- work item: query tile qt of head h in sequence b (high qt first: they have the most work) ----
  const int h = blockIdx.x % p.H_q;
  const int rest = blockIdx.x / p.H_q;
  const int b = rest % p.B;
  const int qt = p.n_tiles - 1 - rest / p.B;
  int seq_start, seq_len;
  if (!seq_bounds(p, b, seq_start, seq_len)) {
    if (threadIdx.x == 0 && qt == p.n_tiles - 1 && h == 0) tg::report(p.status, TG_DEV_BAD_SEQLENS);
    return;
  }
  const int q0 = qt * kTile;
  if (q0 >= seq_len) return;  // uniform for the CTA
  const int n_kv = qt + 1;
  const int kvh = h / p.group;

  if (threadIdx.x == 0) {
    tg::mbar_init(qd_full, 1);
    for (int s = 0; s < C::kStages; ++s) {
      tg::mbar_init(&ring_full[s], 1);
      tg::mbar_init(&ring_empty[s], 1);
    }
    tg::mbar_init(st_full, 1);
    tg::mbar_init(s_free, 8);
    tg::mbar_init(&p_full[0], 8);
    tg::mbar_init(&p_full[1], 8);
    tg::mbar_init(dq_done, 1);
    tg::mbar_init(acc_final, 1);
    for (int s = 0; s < 2; ++s) {
      tg::mbar_init(&col_full[s], 32);
      tg::mbar_init(&col_empty[s], 8);
    }
    tg::mbar_init(drain, 1);
    for (int i = 0; i < 4; ++i) flags[i] = 0;
    tg::fence_mbar_init();
    tg::prefetch_tensormap(&tm_q);
    tg::prefetch_tensormap(&tm_k);
    tg::prefetch_tensormap(&tm_v);
    tg::prefetch_tensormap(&tm_do);
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
      // ---------------- TMA: Q, dO of the query tile once; then (K, V) of every key tile ----------------
      tg::mbar_arrive_expect_tx(qd_full, 2 * C::kTileBytes);
      for (int hf = 0; hf < C::kHalves; ++hf) {
        tg::tma_load_3d(sQ + hf * 16384, &tm_q, qd_full, hf * 64, h, seq_start + q0);
        tg::tma_load_3d(sdO + hf * 16384, &tm_do, qd_full, hf * 64, h, seq_start + q0);
      }
      flags[3] = 1;
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % C::kStages;
        if (!tg::mbar_wait(&ring_empty[s], ((j / C::kStages) & 1) ^ 1u, vabort, p.wait_limit)) {
          *vabort = 1;
          break;
        }
        uint8_t *dst = sRing + s * 2 * C::kTileBytes;
        tg::mbar_arrive_expect_tx(&ring_full[s], 2 * C::kTileBytes);
        for (int hf = 0; hf < C::kHalves; ++hf) {
          tg::tma_load_3d(dst + hf * 16384, &tm_k, &ring_full[s], hf * 64, kvh, seq_start + j * kTile);
          tg::tma_load_3d(dst + C::kTileBytes + hf * 16384, &tm_v, &ring_full[s], hf * 64, kvh,
                          seq_start + j * kTile);
        }
        flags[1] = j + 1;
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issue (converged warp, elected lane) ----------------
    // Software-pipelined: S(j + 1) and dP(j + 1) are issued once the elementwise warps hold S(j) in
    // registers (dP alternates between two column blocks), so they run while c dX(j) is computed;
    // dQ(j) follows c dX(j).
    const uint32_t idesc_st = tg::idesc_bf16_f32(kTile, kTile);     // Q K^T, dO V^T: both K-major
    const uint32_t idesc_acc = tg::idesc_bf16_f32(kTile, D, 0, 1);  // dX K: B MN-major
    const uint64_t dq0 = tg::smem_desc(tg::smem_u32(sQ), 16, 1024, tg::kSwz128);
    const uint64_t ddo0 = tg::smem_desc(tg::smem_u32(sdO), 16, 1024, tg::kSwz128);
    const uint64_t dr0 = tg::smem_desc(tg::smem_u32(sRing), 16, 1024, tg::kSwz128);
    const uint64_t dr0_mn = tg::smem_desc(tg::smem_u32(sRing), 16384, 1024, tg::kSwz128);
    constexpr uint32_t kTile16 = C::kTileBytes >> 4;
    bool ok = __all_sync(0xFFFFFFFFu, tg::mbar_wait(qd_full, 0, vabort, p.wait_limit));
    int consumed = 0;
    for (int j = 0; j <= n_kv && ok; ++j) {
      if (j < n_kv) {
        const int s = j % C::kStages;
        const uint64_t k_off = 2 * s * kTile16, v_off = k_off + kTile16;
        // S(j) overwrites S(j - 1): after the elementwise warps have read it
        ok = __all_sync(0xFFFFFFFFu, tg::mbar_wait(&ring_full[s], (j / C::kStages) & 1, vabort, p.wait_limit));
        if (ok && j > 0) ok = __all_sync(0xFFFFFFFFu, tg::mbar_wait(s_free, (j - 1) & 1, vabort, p.wait_limit));
        if (!ok) break;
        consumed = j + 1;
        tg::tc_fence_after();
        mma_tile_ss<D>(tmem + C::kColS, dq0, dr0 + k_off, idesc_st);
        if (j >= 2) {  // dP(j) overwrites c dX(j - 2): after dQ(j - 2) has read it
          ok = __all_sync(0xFFFFFFFFu, tg::mbar_wait(dq_done, (j - 2) & 1, vabort, p.wait_limit));
          if (!ok) break;
          tg::tc_fence_after();
        }
        mma_tile_ss<D>(tmem + C::dp_col(j), ddo0, dr0 + v_off, idesc_st);
        tg::mma_commit_elect(st_full);
      }
      if (j > 0) {
        const int jp = j - 1, sp = jp % C::kStages;
        ok = __all_sync(0xFFFFFFFFu, tg::mbar_wait(&p_full[jp & 1], (jp >> 1) & 1, vabort, p.wait_limit));
        if (!ok) break;
        tg::tc_fence_after();
        mma_tile_ts<D>(tmem + C::kColAcc0, tmem + C::dp_col(jp), dr0_mn + 2 * sp * kTile16, idesc_acc,
                       jp == 0);   // dQ
        tg::mma_commit_elect(dq_done);
        tg::mma_commit_elect(&ring_empty[sp]);
      }
    }
    if (ok) tg::mma_commit_elect(acc_final);
    if (lane == 0) flags[2] = consumed;
    if (!ok) {
      *vabort = 1;
      tg::mma_commit_elect(drain);
      volatile int32_t never = 0;
      tg::mbar_wait(drain, 0, &never, p.drain_limit);
    }
  } else if (warp == 2) {
    // ---------------- column producer: beta_h log2 g_j of the key tile's 128 keys ----------------
    const float beta = p.beta[h];
    const int gcol = h / p.g_group;
    for (int j = 0; j < n_kv; ++j) {
      const int slot = j & 1;
      if (!tg::mbar_wait(&col_empty[slot], ((j >> 1) & 1) ^ 1u, vabort, p.wait_limit)) {
        *vabort = 1;
        break;
      }
      float *dst = sCols + slot * 256;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = lane * 4 + u, kj = j * kTile + c;
        float v = 0.0f;  // keys past the sequence sit only in the diagonal tile, after every valid query
        if (p.g != nullptr && beta != 0.0f && kj < seq_len) {
          const float lg = tg::log2_gate(p.g[static_cast<size_t>(seq_start + kj) * p.g_cols + gcol]);
          v = beta * lg;
        }
        dst[c] = v;
      }
      tg::mbar_arrive(&col_full[slot]);
    }
  } else if (warp >= 4) {
    // ---------------- elementwise: thread = query row, warps 4-7 / 8-11 = key columns 0-63 / 64-127 ----------------
    const int wq = warp & 3, hh = (warp - 4) >> 2;
    const int r = wq * 32 + lane, qi = q0 + r;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const float ch = p.scale[h], c2 = ch * kLog2e;
    // this row's -LSE log2 e (-inf past the sequence or with no visible weight) and D_i, read from
    // dQ before any CTA writes this row's dQ (only this CTA does, in its epilogue)
    float negl = -INFINITY, dd = 0.0f;
    if (qi < seq_len) {
      const size_t row = static_cast<size_t>(seq_start + qi) * p.H_q + h;
      const float lse = p.lse[row];
      if (lse > -INFINITY) negl = -lse * kLog2e;
      dd = p.dQ[row * D];
    }
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int slot = j & 1;
      const uint32_t dpc = C::dp_col(j);
      bool w = tg::mbar_wait(st_full, j & 1, vabort, p.wait_limit);
      w = w && tg::mbar_wait(&col_full[slot], (j >> 1) & 1, vabort, p.wait_limit);
      ok = barrier_all(1, 256, w);
      if (!ok) break;
      tg::tc_fence_after();
      uint32_t pv[2][32];
      tg::tmem_ld_32x32b_x32(lane_addr + C::kColS + 64 * hh, pv[0]);
      tg::tmem_ld_32x32b_x32(lane_addr + C::kColS + 64 * hh + 32, pv[1]);
      tg::tmem_ld_wait();
      tg::tc_fence_before();
      __syncwarp();
      if (lane == 0) tg::mbar_arrive(s_free);  // S(j) is in registers: S(j + 1) may overwrite it
      const float *bias = sCols + slot * 256;
      const bool diag = j == qt;
      const uint64_t c2x = f2(c2, c2), chx = f2(ch, ch), nlx = f2(negl, negl), ndx = f2(-dd, -dd);
#pragma unroll
      for (int chunk = 0; chunk < 2; ++chunk) {
        const int c0 = 64 * hh + 32 * chunk;
        uint32_t *sv = pv[chunk];
        uint32_t dpv[32], xk[16];
        tg::tmem_ld_32x32b_x32(lane_addr + dpc + c0, dpv);  // lands while P is computed
        const float4 *b4 = reinterpret_cast<const float4 *>(bias + c0);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 bv = b4[c4];
          const uint64_t a = f2_fma(f2(__uint_as_float(sv[4 * c4]), __uint_as_float(sv[4 * c4 + 1])), c2x,
                                    f2_add(nlx, f2(bv.x, bv.y)));
          const uint64_t b = f2_fma(f2(__uint_as_float(sv[4 * c4 + 2]), __uint_as_float(sv[4 * c4 + 3])), c2x,
                                    f2_add(nlx, f2(bv.z, bv.w)));
          float a0, a1, b0, b1;
          f2_split(a, a0, a1);
          f2_split(b, b0, b1);
          sv[4 * c4] = __float_as_uint(a0);
          sv[4 * c4 + 1] = __float_as_uint(a1);
          sv[4 * c4 + 2] = __float_as_uint(b0);
          sv[4 * c4 + 3] = __float_as_uint(b1);
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) sv[c] = __float_as_uint(ex2(__uint_as_float(sv[c])));
        if (diag) {  // key after query: not visible
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (c0 + c > r) sv[c] = 0u;
        }
        tg::tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float s0, s1;
          f2_split(f2_mul(f2_mul(f2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])),
                                 f2_add(f2(__uint_as_float(dpv[c]), __uint_as_float(dpv[c + 1])), ndx)),
                          chx), s0, s1);
          xk[c / 2] = tg::pack_bf16x2(s0, s1);
        }
        tg::tmem_st_32x32b_x16(lane_addr + dpc + 64 * hh + 16 * chunk, xk);
      }
      tg::tmem_st_wait();
      tg::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        tg::mbar_arrive(&p_full[j & 1]);
        tg::mbar_arrive(&col_empty[slot]);
      }
    }
    // ---- epilogue: this row's dQ, half of the D columns per warp group ----
    if (ok) ok = __all_sync(0xFFFFFFFFu, tg::mbar_wait(acc_final, 0, vabort, p.wait_limit));
    if (ok) {
      tg::tc_fence_after();
      // The same staging as the dK / dV pass (Q and dO are idle once acc_final has fired: warp
      // group 0's half rows go to the Q buffer, group 1's to the dO buffer).
      constexpr int kCh = D / 8;  // 16-byte chunks per half row
      float4 *stg = reinterpret_cast<float4 *>(hh == 0 ? sQ : smem + C::kOffFixB);
      for (int c0 = 0; c0 < D / 2; c0 += 32) {
        uint32_t v[32];
        tg::tmem_ld_32x32b_x32(lane_addr + C::kColAcc0 + hh * (D / 2) + c0, v);
        tg::tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 8; ++u)
          stg[r * kCh + ((c0 / 4 + u) ^ (r & (kCh - 1)))] =
              make_float4(__uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]), __uint_as_float(v[4 * u + 2]),
                          __uint_as_float(v[4 * u + 3]));
      }
      __syncwarp();
      const int cl = lane % kCh;
#pragma unroll 4
      for (int rr = 0; rr < 32; rr += 32 / kCh) {
        const int rt = wq * 32 + rr + lane / kCh;  // query row within the tile
        const float4 v = stg[rt * kCh + (cl ^ (rt & (kCh - 1)))];
        if (q0 + rt < seq_len)
          reinterpret_cast<float4 *>(p.dQ + (static_cast<size_t>(seq_start + q0 + rt) * p.H_q + h) * D + hh * (D / 2))[cl] =
              v;
      }
    } else {
      *vabort = 1;
    }
  }

  tg::tc_fence_before();
  __syncthreads();
  if (*vabort) {
    if (threadIdx.x == 0) {
      tg::report(p.status, TG_DEV_TIMEOUT);
      volatile int32_t never = 0;
      for (int i = flags[2]; i < flags[1]; ++i)
        tg::mbar_wait(&ring_full[i % C::kStages], (i / C::kStages) & 1, &never, p.drain_limit);
      if (flags[3]) tg::mbar_wait(qd_full, 0, &never, p.drain_limit);
    }
    __syncthreads();
  }
  if (warp == 1) {
    tg::tc_fence_after();
    tg::tmem_dealloc(tmem, 512);
  }
}

// ---- the gate-score gradient: ds[kept_idx[m], c] = (1 - g[m, c]) sum over the query heads h
// that read gate head c of beta_h dbias[m, h] (one gate head: every h) ----
struct ScoreGradParams {
  const float *dbias, *g_kept;
  const int32_t *kept_idx, *cu_kept;
  int32_t B, capacity, H_q, H_g, T;
  float *ds;
  float beta[kMaxHeads];
};

__global__ void __launch_bounds__(256) gate_score_grad_kernel(const __grid_constant__ ScoreGradParams p) {
  tg::pdl_wait();
  tg::pdl_launch_dependents();
  const int M = max(0, min(p.cu_kept[p.B], p.capacity));
  const int per = p.H_q / p.H_g;
  const long long n = static_cast<long long>(M) * p.H_g;
  for (long long e = blockIdx.x * 256LL + threadIdx.x; e < n; e += gridDim.x * 256LL) {
    const int m = static_cast<int>(e / p.H_g), c = static_cast<int>(e % p.H_g);
    float acc = 0.0f;
    for (int h = c * per; h < (c + 1) * per; ++h)
      acc = fmaf(p.beta[h], p.dbias[static_cast<size_t>(m) * p.H_q + h], acc);
    const int j = p.kept_idx[m];
    if (j >= 0 && j < p.T) p.ds[static_cast<size_t>(j) * p.H_g + c] = acc * (1.0f - p.g_kept[e]);
  }
}

// Tensor maps of the four operands ([M, H, D] bf16, token-major), with the forward's 64 x 1 x 128
// box of 128-byte-swizzled rows.
template <int D>
bool bwd_tensor_maps(const uint16_t *Q, const uint16_t *K, const uint16_t *V, const uint16_t *dO,
                     const BwdParams &p, CUtensorMap *tm) {
  const uint32_t box[3] = {64, 1, kTile};
  const uint16_t *base[4] = {Q, K, V, dO};
  const int heads[4] = {p.H_q, p.H_kv, p.H_kv, p.H_q};
  for (int i = 0; i < 4; ++i) {
    const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(heads[i]),
                              static_cast<uint64_t>(p.M_cap)};
    const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(heads[i]) * D * 2};
    if (!tg_host::encode_tmap_bf16(&tm[i], base[i], 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
  }
  return true;
}

template <int D>
tg_status launch_bwd_d(const uint16_t *Q, const uint16_t *K, const uint16_t *V, const uint16_t *dO,
                       const BwdParams &p, cudaStream_t stream) {
  using C = BwdCfg<D>;
  CUtensorMap tm[4];
  if (!bwd_tensor_maps<D>(Q, K, V, dO, p, tm)) return TG_ERR_CUDA;
  cudaError_t e = cudaFuncSetAttribute(bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return tg_host::record_cuda(e);
  const long long g_kv = static_cast<long long>(p.n_tiles) * p.B * p.H_kv;
  const long long g_q = static_cast<long long>(p.n_tiles) * p.B * p.H_q;
  if (g_q > 0x7FFFFFFFLL) return TG_ERR_UNSUPPORTED;
  long long g_row = (static_cast<long long>(p.M_cap) * p.H_q + 7) / 8;
  const long long cap = static_cast<long long>(tg_host::num_sms()) * 16;
  if (g_row > cap) g_row = cap;
  if (g_row < 1) g_row = 1;
  e = tg_host::launch_pdl(bwd_rowdot_kernel<D>, dim3(static_cast<int>(g_row)), dim3(256), 0, stream, p);
  if (e == cudaSuccess)
    e = tg_host::launch_pdl(bwd_dkdv_kernel<D>, dim3(static_cast<int>(g_kv)), dim3(kThreads), C::kSmemBytes,
                            stream, tm[0], tm[1], tm[2], tm[3], p);
  if (e == cudaSuccess)
    e = tg_host::launch_pdl(bwd_dq_kernel<D>, dim3(static_cast<int>(g_q)), dim3(kThreads), C::kSmemBytes,
                            stream, tm[0], tm[1], tm[2], tm[3], p);
  return tg_host::record_cuda(e);
}

}  // namespace

namespace tg_host {

tg_status launch_gated_attention_bwd(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                                     const float *g, int32_t H_g, const uint16_t *O, const uint16_t *dO,
                                     const float *lse, const int32_t *cu_kept, int32_t B, int32_t M_cap,
                                     int32_t max_seqlen, int32_t H_q, int32_t H_kv, int32_t d_h,
                                     const float *tau, const float *beta, float *dQ, float *dK, float *dV,
                                     float *dbias, int32_t *status, cudaStream_t stream) {
  if (M_cap == 0 || max_seqlen == 0) return TG_OK;
  BwdParams p;
  p.O = O;
  p.dO = dO;
  p.g = g;
  p.g_cols = H_g;
  p.g_group = H_q / H_g;
  p.lse = lse;
  p.cu_kept = cu_kept;
  p.B = B;
  p.M_cap = M_cap;
  p.max_seqlen = max_seqlen;
  p.H_q = H_q;
  p.H_kv = H_kv;
  p.group = H_q / H_kv;
  p.n_tiles = (max_seqlen + kTile - 1) / kTile;
  p.dQ = dQ;
  p.dK = dK;
  p.dV = dV;
  p.dbias = dbias;
  p.status = status;
  p.wait_limit = wait_limit_ns();
  p.drain_limit = drain_limit_ns();
  p.withhold = (withhold_mask() & TG_WITHHOLD_BACKWARD) != 0;
  for (int h = 0; h < kMaxHeads; ++h) {
    p.scale[h] = h < H_q ? tau[h] / std::sqrt(static_cast<float>(d_h)) : 0.0f;
    p.beta[h] = h < H_q ? beta[h] : 0.0f;
  }
  if (d_h == 128) return launch_bwd_d<128>(Q, K, V, dO, p, stream);
  if (d_h == 64) return launch_bwd_d<64>(Q, K, V, dO, p, stream);
  return TG_ERR_UNSUPPORTED;
}

tg_status launch_gate_score_grad(const float *dbias, const float *beta, const float *g_kept, int32_t H_g,
                                 const int32_t *kept_idx, const int32_t *cu_kept, int32_t B,
                                 int32_t capacity, int32_t H_q, int32_t T, float *ds, cudaStream_t stream) {
  if (capacity == 0) return TG_OK;
  ScoreGradParams p;
  p.dbias = dbias;
  p.g_kept = g_kept;
  p.kept_idx = kept_idx;
  p.cu_kept = cu_kept;
  p.B = B;
  p.capacity = capacity;
  p.H_q = H_q;
  p.H_g = H_g;
  p.T = T;
  p.ds = ds;
  for (int h = 0; h < kMaxHeads; ++h) p.beta[h] = h < H_q ? beta[h] : 0.0f;
  int grid = static_cast<int>((static_cast<long long>(capacity) * H_g + 255) / 256);
  if (grid > num_sms() * 4) grid = num_sms() * 4;
  return record_cuda(launch_pdl(gate_score_grad_kernel, dim3(grid), dim3(256), 0, stream, p));
}

}  // namespace tg_host
