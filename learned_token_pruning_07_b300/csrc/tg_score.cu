// tg_score.cu — gate scoring (TokenGate deep dive, section 3.1, Eq. (3): b~_j = MLP(a~_j)).
//
//   u = W1 h_j (+ b1),  s_j = w2 . SiLU(u) (+ b2),  g_j = sigmoid(s_j)  (g = 1 on non-prunable rows)
//
// Persistent kernel on CTA pairs (one CTA per SM): a pair walks 256-row tiles of h (pair tile =
// pair index + k * pairs). The d_g-wide hidden layer of a tile is computed as n_items column
// slices of at most 256 (two slices of 256 at d_g = 512). A slice is one accumulator unit: a
// d-reduction u_slice = h_tile W1_slice^T issued as 2-SM tensor-core MMAs
// (tcgen05.mma.cta_group::2 kind::f16, M = 256): CTA r of the pair stages its own 128 rows of the
// h tile and its half (rows r * item_n / 2 ..) of the W1 slice, and the tensor cores of the two
// SMs share the W1 halves, so each SM takes in 32 KB per K-stage of 64 instead of 48 KB. (With
// every SM loading at once, shared memory fills at about 60 B/clk per SM on this part, under the
// 94 B/clk that one-CTA 128 x 256 tiles would need to keep their MMAs busy.) The accumulator of
// a CTA's 128 rows is in its own tensor memory, in one of two 256-column buffers: the epilogue of
// a unit (SiLU, the w2 dot, and at a tile's last slice the sigmoid) runs while the tensor cores
// already work on the next unit in the other buffer.
//
// With two slices and few tiles for many SMs, the launch uses clusters of four instead: the two
// pairs of a cluster take the two slices of the same tile side by side, and slice 1's CTA hands
// its rows' partial w2 dots to slice 0's CTA with asynchronous remote stores.
//
// Every partial w2 dot of a row is added in a fixed order (column halves, then slices), so s
// is deterministic, and no global scratch memory is needed.
//
// Warp roles (320 threads): warp 0 lane 0 of each CTA issues that CTA's TMA loads, which complete
// on the pair leader's stage barrier; warp 1 owns tensor memory (allocated for the pair), and in
// the leader issues the MMAs (the warp runs converged and one elected lane issues) and commits
// their completion to the barriers of both CTAs; warps 2-9 run the epilogue, two per
// tensor-memory lane quarter (warp w reads lanes 32*(w%4) .. +31, one row per thread, half of
// the columns each), and report a drained accumulator to the leader. With the fused RMSNorm,
// warps 2-5 run the epilogue over all columns and warps 6-9 sum each row's squares. Every wait
// is bounded (see tg_set_wait_limit_ns); a wait that gives up raises the abort flag in every CTA
// of the cluster and sets TG_DEV_TIMEOUT; the CTAs drain the copies and MMAs in flight, free
// tensor memory and return.
#include <mutex>
#include <vector>

#include "tg_common.cuh"

namespace {

constexpr int kBM = 128;      // rows per tile = tensor-memory lanes
constexpr int kBK = 64;       // d-elements per pipeline stage (one 128-byte swizzled row)
// Pipeline stages: 7 with one gate head (b1 and w2 are then read through L1, leaving shared
// memory to the stages), 6 with several (their W2 table stays in shared memory).
__host__ __device__ constexpr int stages_for(int ghp) { return ghp == 1 ? 7 : 6; }
// Warps 0 (TMA), 1 (MMA), 2-9: eight epilogue warps (two per tensor-memory lane quarter, each
// taking half of every slice's columns), or with the fused RMSNorm four epilogue warps (2-5)
// and four that sum each row's squares (6-9).
constexpr int kThreads = 320;
__host__ __device__ constexpr int epi_warps(bool norm) { return norm ? 4 : 8; }
constexpr int kMaxDg = 512;
constexpr int kMaxItemN = 256;  // columns of one slice = one MMA N = one accumulator buffer
constexpr uint32_t kTmemCols = 2 * kMaxItemN;
constexpr int kMaxGateHeads = 16;
constexpr int kPair = 2;  // CTAs of a cluster: the two halves (128 rows each) of a 256-row tile
// Barrier region: full, empty and landed per stage (at most 7 stages), acc_full[2], acc_empty[2],
// drain, rms_ready[2], rms_free[2], xch_full[4], xch_free[4], xq_full[4], xq_free[4]; then the
// tensor-memory slot, three int32 flags and four reply words.
constexpr uint32_t kBarBytes = 400;
constexpr int kMaxQuadHeads = 8;  // padded gate heads up to which clusters of four are used
constexpr uint32_t kSmemLimit = 232448;  // dynamic shared memory a CTA may opt into
static_assert((3 * 7 + 9 + 8 + 8) * 8 + 4 * 4 + 4 * 4 <= kBarBytes, "barrier region too small");

struct ScoreParams {
  int32_t T, d, d_g, n_items, item_n, n_tiles, KT;  // n_tiles: 256-row pair tiles
  float ln_eps;  // fused RMSNorm (LN_2 of the residual): 1 / sqrt(mean(h^2) + ln_eps) per row
  const float *b1;
  const uint16_t *w2;  // [H_g, d_g] (one row per gate head)
  float b2;
  int32_t H_g;                  // gate heads (section 3.4: a per-head bias), <= kMaxGateHeads
  float b2h[kMaxGateHeads];     // per-head second-layer bias (H_g > 1)
  const uint8_t *mask;
  float *s_out;  // [T, H_g]
  float *g_out;  // [T, H_g] or NULL
  float *s_sel;  // H_g > 1: [T] uniform head aggregation (the row mean) that top-K ranks
  int32_t *status;
  uint64_t wait_limit, drain_limit;
  int32_t withhold;  // test hook: 1: no CTA issues its loads; 2: CTAs of odd cluster rank issue none
  int32_t quad;      // clusters of four: the two pairs of a cluster take the two slices of a tile
};

__device__ const float g_zero_b1[kMaxDg] = {};  // b1 of a layer without a first-layer bias

struct SmemLayout {
  uint32_t a_bytes, b_bytes, off_b, off_w2, off_b1, off_rms, off_xq, off_bar, total;
};

// ghp: gate heads padded to 1, 2, 4, 8 or 16. More than one head keeps W2 as bf16 pairs
// [d_g][ghp / 2] (16 KB at 16 heads, zero past H_g) and b1 as fp32 [d_g] in shared memory.
__host__ __device__ inline SmemLayout score_smem_layout(int item_n, int ghp, bool norm) {
  SmemLayout L;
  const int S = stages_for(ghp);
  L.a_bytes = kBM * kBK * 2;                               // 16 KB
  L.b_bytes = static_cast<uint32_t>(item_n / kPair) * kBK * 2;  // this CTA's half: <= 16 KB
  L.off_b = S * L.a_bytes;
  L.off_w2 = L.off_b + S * L.b_bytes;
  L.off_b1 = L.off_w2 + (ghp == 1 ? 0 : kMaxDg * ghp * 2);
  // fused RMSNorm: [2 tiles][128 rows] fp32 1 / rms; otherwise [ghp][128 rows] fp32, the
  // second-half epilogue warps' partial row sums handed to the first half
  L.off_rms = L.off_b1 + (ghp == 1 ? 0 : kMaxDg * 4);
  L.off_xq = L.off_rms + (norm ? 2 * kBM * 4 : kBM * ghp * 4);
  // [ghp][128 rows] fp32: slice 1's partial sums (clusters of four, at most 8 heads: 16 heads
  // leave no room for it beside six stages)
  L.off_bar = L.off_xq + (ghp <= kMaxQuadHeads ? kBM * ghp * 4 : 0);
  L.total = L.off_bar + kBarBytes + 1024;  // barriers + slots, plus alignment slack
  return L;
}

// ---- the CTA pair: cluster addresses, TMA into this CTA completing on the leader's barrier,
// 2-SM MMAs, commits to a barrier of either CTA, and the pair's tensor memory ----

// Address of this CTA's shared variable `p` in the shared memory of CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void *p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(tg::smem_u32(p)), "r"(rank));
  return r;
}

__device__ __forceinline__ void tma_load_2d_to_leader(void *dst, const CUtensorMap *map, uint32_t bar_cluster,
                                                      int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(tg::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void mma2_bf16_ss_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                   uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One arrival on the barrier at `bar_cluster` (either CTA) once every 2-SM MMA issued so far by
// the elected lane has completed.
__device__ __forceinline__ void commit2_elect(uint32_t bar_cluster) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar_cluster)
      : "memory");
}

// A 4-byte store into the shared memory of another CTA of the cluster that, once it lands,
// completes 4 bytes of the transaction count of the barrier at `bar_cluster` (in that CTA).
__device__ __forceinline__ void st_async_b32(uint32_t addr_cluster, uint32_t v, uint32_t bar_cluster) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(addr_cluster),
               "r"(v), "r"(bar_cluster)
               : "memory");
}

// Raise the abort flag in every CTA of the cluster (a plain store into each one's shared
// memory), so that all of them stop issuing and leave their waits together.
__device__ __forceinline__ void raise_abort(int32_t *abort_flag, uint32_t crank, int csize) {
  *reinterpret_cast<volatile int32_t *>(abort_flag) = 1;
  for (int r = 0; r < csize; ++r)
    if (static_cast<uint32_t>(r) != crank)
      asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr(abort_flag, static_cast<uint32_t>(r))), "r"(1)
                   : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Tensor memory for 2-SM MMAs: a warp of each CTA of the pair runs these together.
__device__ __forceinline__ void tmem_alloc2(uint32_t *dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tg::smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Epilogue of NC accumulator columns of one row (hidden units hid .. hid + NC - 1): u = the
// accumulator (times 1 / rms under the fused RMSNorm) + b1, then w2 . SiLU(u) into acc (one
// head) or, per head pair, into the packed fp32 pairs acc2, in column order.
// b1: fp32 [d_g] (global memory with one head, read through L1; shared memory otherwise);
// w2g: the one head's bf16 w2 [d_g] in global memory; s_w2h: the heads' bf16 pairs in shared memory.
template <int NC, bool NORM, int GHP>
__device__ __forceinline__ void score_chunk(const uint32_t (&v)[NC], int hid, float inv_rms, const float *b1,
                                            const uint16_t *w2g, const uint32_t *s_w2h, float *acc, uint64_t *acc2) {
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    const float bias = GHP == 1 ? __ldg(b1 + hid + i) : b1[hid + i];
    const float u = NORM ? fmaf(__uint_as_float(v[i]), inv_rms, bias) : __uint_as_float(v[i]) + bias;
    const float silu = __fdividef(u, 1.0f + __expf(-u));
    if constexpr (GHP == 1) {
      acc[0] = fmaf(tg::bf16_bits_to_float(__ldg(w2g + hid + i)), silu, acc[0]);
    } else {
      // every thread reads the same column's weights: a shared-memory broadcast
      uint32_t w[GHP / 2];
      const uint32_t *src = s_w2h + (hid + i) * (GHP / 2);
      if constexpr (GHP >= 8) {
#pragma unroll
        for (int k = 0; k < GHP / 2; k += 4) {
          const uint4 q = *reinterpret_cast<const uint4 *>(src + k);
          w[k] = q.x; w[k + 1] = q.y; w[k + 2] = q.z; w[k + 3] = q.w;
        }
      } else {
#pragma unroll
        for (int k = 0; k < GHP / 2; ++k) w[k] = src[k];
      }
      uint64_t silu2;
      asm("mov.b64 %0, {%1, %1};" : "=l"(silu2) : "f"(silu));
#pragma unroll
      for (int k = 0; k < GHP / 2; ++k) {
        uint64_t wk;  // the bf16 pair widened to fp32: low half, then high half
        asm("mov.b64 %0, {%1, %2};" : "=l"(wk) : "r"(w[k] << 16), "r"(w[k] & 0xFFFF0000u));
        asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2[k]) : "l"(wk), "l"(silu2));
      }
    }
  }
}

template <bool NORM, int GHP>
__global__ void __launch_bounds__(kThreads, 1)
    gate_score_kernel(const __grid_constant__ CUtensorMap tm_h,
                      const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ ScoreParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const SmemLayout L = score_smem_layout(p.item_n, GHP, NORM);
  constexpr int EW = epi_warps(NORM);
  uint8_t *sA = smem;
  uint8_t *sB = smem + L.off_b;
  uint32_t *s_w2h = reinterpret_cast<uint32_t *>(smem + L.off_w2);  // GHP > 1: [d_g][GHP / 2] bf16 pairs
  float *s_b1 = reinterpret_cast<float *>(smem + L.off_b1);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.off_bar);
  constexpr int kStages = stages_for(GHP);
  uint64_t *empty = full + kStages;
  uint64_t *acc_full = empty + kStages;  // [2] MMA -> epilogue
  uint64_t *acc_empty = acc_full + 2;    // [2] epilogue -> MMA
  uint64_t *drain = acc_empty + 2;
  uint64_t *rms_ready = drain + 1;       // [2] norm warps -> epilogue (by tile parity)
  uint64_t *rms_free = rms_ready + 2;    // [2] epilogue -> norm warps
  float *s_inv_rms = reinterpret_cast<float *>(smem + L.off_rms);
  uint64_t *landed = rms_free + 2;       // [kStages] leader's MMA commit -> the peer's norm warps
  uint64_t *xch_full = landed + kStages;  // [4] per lane quarter: second-half partial sums written
  uint64_t *xch_free = xch_full + 4;      // [4] per lane quarter: the first half has read them
  float *s_xch = s_inv_rms;               // without the fused RMSNorm: [GHP][128 rows] partial sums
  uint64_t *xq_full = xch_free + 4;       // [4] clusters of four: slice 1's partial sums landed here
  uint64_t *xq_free = xq_full + 4;        // [4] slice 0's CTA has read them (its reply landed here)
  float *s_xq = reinterpret_cast<float *>(smem + L.off_xq);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(xq_free + 4);
  int32_t *abort_flag = reinterpret_cast<int32_t *>(tmem_slot + 1);
  int32_t *n_issued = abort_flag + 1;
  int32_t *n_consumed = abort_flag + 2;
  uint32_t *xq_word = reinterpret_cast<uint32_t *>(n_consumed + 1);  // [4] targets of the replies

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint32_t crank;
  asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(crank));
  const uint32_t rank = crank & 1u;       // position in the CTA pair (peer CTAs differ in bit 0)
  const uint32_t pb = crank & ~1u;        // cluster rank of the pair's leader
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      tg::mbar_init(&full[i], 1);  // the leader's: its own expect_tx, the bytes of both CTAs
      // one MMA commit from the leader (+ this CTA's four norm warps)
      tg::mbar_init(&empty[i], 1 + (NORM ? 4 : 0));
    }
    for (int i = 0; i < 2; ++i) {
      tg::mbar_init(&acc_full[i], 1);
      tg::mbar_init(&acc_empty[i], EW * kPair);  // the leader's: every epilogue warp of both CTAs
    }
    tg::mbar_init(drain, 1);
    for (int i = 0; i < 2; ++i) {
      tg::mbar_init(&rms_ready[i], 4);
      tg::mbar_init(&rms_free[i], 4);
    }
    for (int i = 0; i < kStages; ++i) tg::mbar_init(&landed[i], 1);
    for (int i = 0; i < 4; ++i) {
      tg::mbar_init(&xch_full[i], 1);
      tg::mbar_init(&xch_free[i], 1);
      tg::mbar_init(&xq_full[i], 1);
      tg::mbar_init(&xq_free[i], 1);
    }
    *abort_flag = 0;
    *n_issued = 0;
    *n_consumed = 0;
    tg::fence_mbar_init();
    tg::prefetch_tensormap(&tm_h);
    tg::prefetch_tensormap(&tm_w);
  }
  if (warp == 1) {
    tmem_alloc2(tmem_slot, kTmemCols);
    tmem_relinquish2();
  }
  tg::pdl_wait();
  tg::pdl_launch_dependents();
  if constexpr (GHP > 1) {
    for (int i = threadIdx.x; i < p.d_g; i += blockDim.x) {
#pragma unroll
      for (int k = 0; k < GHP / 2; ++k) {
        const uint32_t lo = 2 * k < p.H_g ? p.w2[static_cast<size_t>(2 * k) * p.d_g + i] : 0u;
        const uint32_t hi = 2 * k + 1 < p.H_g ? p.w2[static_cast<size_t>(2 * k + 1) * p.d_g + i] : 0u;
        s_w2h[i * (GHP / 2) + k] = lo | (hi << 16);
      }
      s_b1[i] = p.b1 ? p.b1[i] : 0.0f;
    }
  }
  // one head: b1 (or zeros) and w2 straight from global memory
  const float *b1_src = GHP == 1 ? (p.b1 ? p.b1 : g_zero_b1) : s_b1;
  tg::tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers are initialised before any remote arrival
  tg::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  volatile int32_t *vabort = abort_flag;
  // The 2-SM MMAs write the peer's accumulator at the leader's address: the pair's allocations
  // must agree (otherwise no work is done and the launch reports TG_DEV_TIMEOUT).
  bool tmem_ok;
  {
    uint32_t other;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(other) : "r"(cluster_addr(tmem_slot, crank ^ 1u)));
    tmem_ok = other == tmem;
    if (!tmem_ok && threadIdx.x == 0) *vabort = 1;
  }
  // both halves of every stage land on the leader's full barrier
  const uint32_t stage_bytes = kPair * (L.a_bytes + L.b_bytes);
  // a cluster is one pair, or (p.quad) two pairs that share each tile: pair crank / 2 takes slice
  // crank / 2 of it, so a tile is one accumulator unit per pair instead of n_items
  const int csize = p.quad ? 2 * kPair : kPair;
  const int tile0 = blockIdx.x / csize;
  const int tile_stride = gridDim.x / csize;
  const int item_lo = p.quad ? static_cast<int>(crank >> 1) : 0;
  const int item_hi = p.quad ? item_lo + 1 : p.n_items;
  const int half_n = p.item_n / kPair;  // W1 rows of a slice this CTA stages

  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer: stage = h tile [128 x 64] + W1 slice [item_n x 64] ----
      int kc = 0;
      bool ok = tmem_ok && !(p.withhold == 1 || (p.withhold == 2 && (crank & 1u)));
      for (int tile = tile0; tile < p.n_tiles && ok; tile += tile_stride) {
        for (int item = item_lo; item < item_hi && ok; ++item) {
          for (int kt = 0; kt < p.KT; ++kt, ++kc) {
            const int st = kc % kStages;
            if (!tg::mbar_wait(&empty[st], ((kc / kStages) & 1) ^ 1u, vabort, p.wait_limit)) {
              raise_abort(abort_flag, crank, csize);
              ok = false;
              break;
            }
            // this CTA's 128 rows of the 256-row h tile and its half of the W1 slice, completing on
            // the leader's barrier (the leader announces the bytes of both CTAs)
            if (leader) tg::mbar_arrive_expect_tx(&full[st], stage_bytes);
            const uint32_t bar = cluster_addr(&full[st], pb);
            tma_load_2d_to_leader(sA + st * L.a_bytes, &tm_h, bar, kt * kBK, tile * (kPair * kBM) + rank * kBM);
            tma_load_2d_to_leader(sB + st * L.b_bytes, &tm_w, bar, kt * kBK, item * p.item_n + rank * half_n);
            *n_issued = kc + 1;
          }
        }
      }
      // tail: the leader's last commits to this CTA's stage barriers have landed before it exits
      for (int k = kc - kStages < 0 ? 0 : kc - kStages; ok && k < kc; ++k)
        ok = tg::mbar_wait(&empty[k % kStages], (k / kStages) & 1, vabort, p.wait_limit);
      if (!ok) raise_abort(abort_flag, crank, csize);
    }
  } else if (warp == 1) {
    if (leader) {
      // ---- MMA issuer (converged warp, elected lane):
      //      u_slice[256 x item_n] += A[256 x 16] * B[item_n x 16]^T over the pair ----
      const uint32_t idesc = tg::idesc_bf16_f32(kPair * kBM, p.item_n);
      const uint64_t a0 = tg::smem_desc(tg::smem_u32(sA), 16, 1024, tg::kSwz128);
      const uint64_t b0 = tg::smem_desc(tg::smem_u32(sB), 16, 1024, tg::kSwz128);
      int kc = 0, it = 0;
      bool ok = tmem_ok;
      for (int tile = tile0; tile < p.n_tiles && ok; tile += tile_stride) {
        for (int item = item_lo; item < item_hi && ok; ++item, ++it) {
          const int buf = it & 1;
          if (!__all_sync(0xFFFFFFFFu, tg::mbar_wait(&acc_empty[buf], ((it >> 1) & 1) ^ 1u, vabort, p.wait_limit))) {
            ok = false;
            break;
          }
          tg::tc_fence_after();
          const uint32_t d_tmem = tmem + buf * kMaxItemN;
          for (int kt = 0; kt < p.KT; ++kt, ++kc) {
            const int st = kc % kStages;
            if (!__all_sync(0xFFFFFFFFu, tg::mbar_wait(&full[st], (kc / kStages) & 1, vabort, p.wait_limit))) {
              ok = false;
              break;
            }
            tg::tc_fence_after();
            const uint64_t ad = a0 + ((st * L.a_bytes) >> 4), bd = b0 + ((st * L.b_bytes) >> 4);
#pragma unroll
            for (int ks = 0; ks < kBK / 16; ++ks)  // a K-step of 16 is 32 bytes into the 128-byte row
              mma2_bf16_ss_elect(d_tmem, ad + 2 * ks, bd + 2 * ks, idesc, (kt | ks) != 0);
            // the peer's norm warps may read their half once these MMAs have (a release arrival to
            // another CTA would cost this thread about 2,000 cycles; a commit costs it nothing)
            if (NORM) commit2_elect(cluster_addr(&landed[st], pb | 1u));
            // the stage is free in both CTAs once these MMAs have read it
            commit2_elect(cluster_addr(&empty[st], pb));
            commit2_elect(cluster_addr(&empty[st], pb | 1u));
            if (lane == 0) *n_consumed = kc + 1;
          }
          if (ok) {
            commit2_elect(cluster_addr(&acc_full[buf], pb));
            commit2_elect(cluster_addr(&acc_full[buf], pb | 1u));
          }
        }
      }
      if (!ok) {
        raise_abort(abort_flag, crank, csize);
        // drain: wait for the MMAs already issued before the tiles and TMEM go away
        commit2_elect(cluster_addr(drain, pb));
        volatile int32_t never = 0;
        tg::mbar_wait(drain, 0, &never, p.drain_limit);
      }
    }
  } else if (warp < 2 + EW) {
    // ---- epilogue: one row per thread; SiLU . w2 over each slice, sigmoid at the end ----
    const int quarter = warp & 3;  // tensor-memory lane quarter this warp may read
    const int half = (warp - 2) >> 2;  // with eight epilogue warps: which half of the columns
    const int r = quarter * 32 + lane;
    // this warp's 16-column groups of every slice
    const int n_g = p.item_n >> 4;
    const int g0 = (EW == 8 && half == 1) ? n_g / 2 : 0;
    const int g1 = (EW == 8 && half == 0) ? n_g / 2 : n_g;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    // accumulator units (tile, slice) this pair computes
    const int n_units = tile0 < p.n_tiles ? ((p.n_tiles - 1 - tile0) / tile_stride + 1) * (item_hi - item_lo) : 0;
    int it = 0, ti = 0;
    bool ok = tmem_ok;
    for (int tile = tile0; tile < p.n_tiles && ok; tile += tile_stride, ++ti) {
      float acc[GHP];
#pragma unroll
      for (int c = 0; c < GHP; ++c) acc[c] = 0.0f;
      uint64_t acc2[GHP > 1 ? GHP / 2 : 1];  // head pairs (2k, 2k + 1) as packed fp32
#pragma unroll
      for (int k = 0; k < (GHP > 1 ? GHP / 2 : 1); ++k) acc2[k] = 0ull;
      float inv_rms = 1.0f;
      if (NORM) {
        ok = __all_sync(0xFFFFFFFFu, tg::mbar_wait(&rms_ready[ti & 1], (ti >> 1) & 1, vabort, p.wait_limit));
        if (!ok) break;
        inv_rms = s_inv_rms[(ti & 1) * kBM + r];
      }
      for (int item = item_lo; item < item_hi; ++item, ++it) {
        const int buf = it & 1;
        // tcgen05.ld is warp-collective: the whole warp takes the same branch
        ok = __all_sync(0xFFFFFFFFu, tg::mbar_wait(&acc_full[buf], (it >> 1) & 1, vabort, p.wait_limit));
        if (!ok) break;
        tg::tc_fence_after();
        const uint32_t taddr = lane_base + static_cast<uint32_t>(buf * kMaxItemN);
        const int hid0 = item * p.item_n;
        // 32-column chunks over this warp's groups; an odd group count ends with a 16-column
        // chunk (a 32-column load there would take in columns that are not this warp's)
        int g = g0;
        for (; g + 2 <= g1; g += 2) {
          uint32_t v[32];
          tg::tmem_ld_32x32b_x32(taddr + g * 16, v);
          tg::tmem_ld_wait();
          score_chunk<32, NORM, GHP>(v, hid0 + g * 16, inv_rms, b1_src, p.w2, s_w2h, acc, acc2);
        }
        if (g < g1) {
          uint32_t vt[16];
          tg::tmem_ld_32x32b_x16(taddr + g * 16, vt);
          tg::tmem_ld_wait();
          score_chunk<16, NORM, GHP>(vt, hid0 + g * 16, inv_rms, b1_src, p.w2, s_w2h, acc, acc2);
        }
        tg::tc_fence_before();
        __syncwarp();
        // the leader's MMAs may reuse this buffer in both CTAs. The MMAs wait for a buffer only
        // before the unit two ahead, so the last two units need no report; the peer skips them,
        // since a release arrival to another CTA holds its warp for about 2,000 cycles
        if (lane == 0) {
          if (leader) tg::mbar_arrive(&acc_empty[buf]);
          else if (it + 2 < n_units) mbar_arrive_cluster(cluster_addr(&acc_empty[buf], pb));
        }
      }
      if (!ok) break;
      if constexpr (GHP > 1) {
#pragma unroll
        for (int k = 0; k < GHP / 2; ++k)
          asm("mov.b64 {%0, %1}, %2;" : "=f"(acc[2 * k]), "=f"(acc[2 * k + 1]) : "l"(acc2[k]));
      }
      if (NORM) {
        __syncwarp();
        if (lane == 0) tg::mbar_arrive(&rms_free[ti & 1]);  // this tile's 1/rms slots are free
      }
      if constexpr (EW == 8) {
        // the second half hands its partial sums to the first, which adds them after its own
        // (a fixed order, so s does not depend on timing) and writes the row's results
        if (half == 1) {
          ok = __all_sync(0xFFFFFFFFu, tg::mbar_wait(&xch_free[quarter], (ti & 1) ^ 1u, vabort, p.wait_limit));
          if (!ok) break;
#pragma unroll
          for (int c = 0; c < GHP; ++c) s_xch[c * kBM + r] = acc[c];
          __syncwarp();
          if (lane == 0) tg::mbar_arrive(&xch_full[quarter]);
          continue;
        }
        ok = __all_sync(0xFFFFFFFFu, tg::mbar_wait(&xch_full[quarter], ti & 1, vabort, p.wait_limit));
        if (!ok) break;
#pragma unroll
        for (int c = 0; c < GHP; ++c) acc[c] += s_xch[c * kBM + r];
        __syncwarp();
        if (lane == 0) tg::mbar_arrive(&xch_free[quarter]);
      }
      if (GHP <= kMaxQuadHeads && p.quad) {
        // Clusters of four: slice 1's pair hands its partial sums to slice 0's CTA with the same
        // rows (cluster rank crank - 2) as asynchronous remote stores that complete on that CTA's
        // barrier (a release arrival to another CTA would hold this warp for ~2,000 cycles);
        // slice 0 adds them after its own (slice order) and writes the row's results, then
        // replies with one word so the buffer may be refilled.
        if (crank >= 2) {
          if (ti > 0) {
            if (lane == 0) tg::mbar_arrive_expect_tx(&xq_free[quarter], 4u);
            ok = __all_sync(0xFFFFFFFFu, tg::mbar_wait(&xq_free[quarter], (ti - 1) & 1, vabort, p.wait_limit));
            if (!ok) break;
          }
          const uint32_t bar = cluster_addr(&xq_full[quarter], crank - 2);
#pragma unroll
          for (int c = 0; c < GHP; ++c) st_async_b32(cluster_addr(&s_xq[c * kBM + r], crank - 2), __float_as_uint(acc[c]), bar);
          continue;
        }
        if (lane == 0) tg::mbar_arrive_expect_tx(&xq_full[quarter], 32u * GHP * 4u);
        ok = __all_sync(0xFFFFFFFFu, tg::mbar_wait(&xq_full[quarter], ti & 1, vabort, p.wait_limit));
        if (!ok) break;
#pragma unroll
        for (int c = 0; c < GHP; ++c) acc[c] += s_xq[c * kBM + r];
        __syncwarp();
        if (lane == 0 && tile + tile_stride < p.n_tiles)
          st_async_b32(cluster_addr(&xq_word[quarter], crank + 2), 1u, cluster_addr(&xq_free[quarter], crank + 2));
      }
      const int row = tile * (kPair * kBM) + static_cast<int>(rank) * kBM + r;
      if (row < p.T) {
        const bool keep_always = p.mask && p.mask[row];
        if (GHP == 1) {
          const float s = acc[0] + p.b2;
          p.s_out[row] = s;
          if (p.s_sel != nullptr && p.s_sel != p.s_out) p.s_sel[row] = s;  // one head: the mean is s
          if (p.g_out) p.g_out[row] = keep_always ? 1.0f : 1.0f / (1.0f + __expf(-s));
        } else {
          // per-head scores and gates, and their uniform aggregation (head order, then / H_g)
          float sum = 0.0f;
          const size_t base = static_cast<size_t>(row) * p.H_g;
#pragma unroll
          for (int c = 0; c < GHP; ++c) {
            if (c < p.H_g) {
              const float s = acc[c] + p.b2h[c];
              sum += s;
              p.s_out[base + c] = s;
              if (p.g_out) p.g_out[base + c] = keep_always ? 1.0f : 1.0f / (1.0f + __expf(-s));
            }
          }
          p.s_sel[row] = sum / static_cast<float>(p.H_g);
        }
      }
    }
    if (!ok) raise_abort(abort_flag, crank, csize);
  } else if (NORM) {
    // ---- norm warps: sum of squares of each row of the tile as its h stages stream past ----
    // Row r of a 128-byte-swizzled stage holds its eight 16-byte chunks at positions c ^ (r % 8).
    const int r = (warp - 6) * 32 + lane;
    int kc = 0, ti = 0;
    bool ok = tmem_ok;
    for (int tile = tile0; tile < p.n_tiles && ok; tile += tile_stride, ++ti) {
      float sq = 0.0f;
      for (int item = item_lo; item < item_hi && ok; ++item) {
        for (int kt = 0; kt < p.KT; ++kt, ++kc) {
          const int st = kc % kStages;
          // the peer's stages complete on the leader's barrier; its norm warps learn that a stage
          // has landed from the commit of the MMAs that read it
          ok = __all_sync(0xFFFFFFFFu, tg::mbar_wait(leader ? &full[st] : &landed[st], (kc / kStages) & 1, vabort,
                                                     p.wait_limit));
          if (!ok) break;
          if (item == item_lo) {  // every slice re-reads the same h tile; the first pass suffices
            const uint4 *row_base = reinterpret_cast<const uint4 *>(sA + st * L.a_bytes + r * 128);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint4 q = row_base[c ^ (r & 7)];
              const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xFFFF0000u);
                sq = fmaf(lo, lo, sq);
                sq = fmaf(hi, hi, sq);
              }
            }
          }
          __syncwarp();
          if (lane == 0) tg::mbar_arrive(&empty[st]);
        }
        if (ok && item == item_lo) {
          ok = __all_sync(0xFFFFFFFFu,
                          tg::mbar_wait(&rms_free[ti & 1], ((ti >> 1) & 1) ^ 1u, vabort, p.wait_limit));
          if (!ok) break;
          s_inv_rms[(ti & 1) * kBM + r] = 1.0f / sqrtf(sq / static_cast<float>(p.d) + p.ln_eps);
          __syncwarp();
          if (lane == 0) tg::mbar_arrive(&rms_ready[ti & 1]);
        }
      }
    }
    if (!ok) raise_abort(abort_flag, crank, csize);
  }

  tg::tc_fence_before();
  __syncthreads();
  if (*vabort) {
    if (threadIdx.x == 0) {
      tg::report(p.status, TG_DEV_TIMEOUT);
      // wait (bounded) for TMA copies that were issued but never consumed; the copies of both
      // CTAs complete on the leader's barriers
      // (one budget for all of them: when a peer withheld its half, these phases never complete)
      volatile int32_t never = 0;
      if (leader) {
        const uint64_t t0 = tg::globaltimer_ns();
        for (int i = *n_consumed; i < *n_issued; ++i) {
          const uint64_t spent = tg::globaltimer_ns() - t0;
          if (spent >= p.drain_limit) break;
          tg::mbar_wait(&full[i % kStages], (i / kStages) & 1, &never, p.drain_limit - spent);
        }
      }
    }
    __syncthreads();
  }
  // no CTA of the pair frees tensor memory or exits while the other may still arrive on its
  // barriers or run MMAs into its tensor memory
  cluster_sync_all();
  if (warp == 1) {
    tg::tc_fence_after();
    tmem_dealloc2(tmem, kTmemCols);
  }
}

}  // namespace

namespace tg_host {

namespace {

// Clusters of `csize` CTAs that are resident at once for this kernel and shared-memory size
// (cached per device, kernel, size and cluster size; at least one).
cudaError_t resident_clusters(const void *kernel, int threads, size_t smem, int csize, int *clusters) {
  struct Entry {
    int dev;
    const void *kernel;
    size_t smem;
    int csize;
    int clusters;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry &c : cache)
    if (c.dev == dev && c.kernel == kernel && c.smem == smem && c.csize == csize) {
      *clusters = c.clusters;
      return cudaSuccess;
    }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(csize * num_sms());
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
  if (e != cudaSuccess) return e;
  if (n < 1) n = 1;
  cache.push_back({dev, kernel, smem, csize, n});
  *clusters = n;
  return cudaSuccess;
}

// Launch with the cluster size given at run time and programmatic dependent launch.
template <typename... KArgs, typename... Args>
cudaError_t launch_clusters(void (*kernel)(KArgs...), int clusters, int csize, int threads, size_t smem,
                            cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(clusters * csize);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <bool NORM>
decltype(&gate_score_kernel<NORM, 1>) score_kernel_for(int ghp) {
  switch (ghp) {
    case 1: return gate_score_kernel<NORM, 1>;
    case 2: return gate_score_kernel<NORM, 2>;
    case 4: return gate_score_kernel<NORM, 4>;
    case 8: return gate_score_kernel<NORM, 8>;
    default: return gate_score_kernel<NORM, 16>;
  }
}

}  // namespace

tg_status launch_gate_score(const uint16_t *h, int32_t T, int32_t d, const uint8_t *mask,
                            const uint16_t *W1, const float *b1, const uint16_t *w2, float b2,
                            int32_t d_g, float *s_out, float *g_out, int32_t *status,
                            cudaStream_t stream, bool rmsnorm, float ln_eps, int32_t H_g,
                            const float *b2h, float *s_sel) {
  if (T == 0) return TG_OK;
  if (H_g < 1 || H_g > kMaxGateHeads) return TG_ERR_UNSUPPORTED;
  ScoreParams p;
  p.H_g = H_g;
  for (int c = 0; c < kMaxGateHeads; ++c) p.b2h[c] = (b2h != nullptr && c < H_g) ? b2h[c] : 0.0f;
  p.s_sel = s_sel;
  const int ghp = H_g == 1 ? 1 : H_g <= 2 ? 2 : H_g <= 4 ? 4 : H_g <= 8 ? 8 : 16;
  p.T = T;
  p.d = d;
  p.d_g = d_g;
  p.ln_eps = ln_eps;
  p.n_items = d_g > kMaxItemN ? 2 : 1;
  p.item_n = d_g / p.n_items;  // d_g % 32 == 0, so a multiple of 16, at most 256
  p.n_tiles = (T + kPair * kBM - 1) / (kPair * kBM);
  p.KT = (d + kBK - 1) / kBK;  // a ragged last stage reads zeros past d from both operands
  p.b1 = b1;
  p.w2 = w2;
  p.b2 = b2;
  p.mask = mask;
  p.s_out = s_out;
  p.g_out = g_out;
  p.status = status;
  p.wait_limit = wait_limit_ns();
  p.drain_limit = drain_limit_ns();
  p.withhold = (withhold_mask() & TG_WITHHOLD_GATE_SCORE) ? 1 : (withhold_mask() & TG_WITHHOLD_GATE_SCORE_PEER) ? 2 : 0;
  p.quad = 0;

  CUtensorMap tm_h, tm_w;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(d), static_cast<uint64_t>(T)};
    const uint64_t strides[1] = {static_cast<uint64_t>(d) * 2};
    const uint32_t box[2] = {kBK, kBM};
    if (!encode_tmap_bf16(&tm_h, h, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return TG_ERR_CUDA;
  }
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(d), static_cast<uint64_t>(d_g)};
    const uint64_t strides[1] = {static_cast<uint64_t>(d) * 2};
    const uint32_t box[2] = {kBK, static_cast<uint32_t>(p.item_n / kPair)};  // one CTA's half of a slice
    if (!encode_tmap_bf16(&tm_w, W1, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return TG_ERR_CUDA;
  }
  const SmemLayout L = score_smem_layout(p.item_n, ghp, rmsnorm);
  if (L.total > kSmemLimit) return TG_ERR_UNSUPPORTED;
  auto kernel = rmsnorm ? score_kernel_for<true>(ghp) : score_kernel_for<false>(ghp);
  const int threads = kThreads;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
  if (e != cudaSuccess) return record_cuda(e);
  // One wave of clusters: as many as fit at once (a cluster sits in one GPC). Pairs walk the
  // tiles with both slices each; clusters of four, where the two pairs take the two slices of a
  // tile side by side, when that takes fewer slice-rounds (few tiles for many SMs).
  int pairs = 0;
  e = resident_clusters(reinterpret_cast<const void *>(kernel), threads, L.total, kPair, &pairs);
  if (e != cudaSuccess) return record_cuda(e);
  p.quad = 0;
  int csize = kPair, clusters = pairs;
  if (p.n_items == 2 && ghp <= kMaxQuadHeads) {
    int quads = 0;
    e = resident_clusters(reinterpret_cast<const void *>(kernel), threads, L.total, 2 * kPair, &quads);
    if (e != cudaSuccess) return record_cuda(e);
    const int rounds_pair = 2 * ((p.n_tiles + pairs - 1) / pairs);
    const int rounds_quad = (p.n_tiles + quads - 1) / quads;
    if (rounds_quad < rounds_pair) {
      p.quad = 1;
      csize = 2 * kPair;
      clusters = quads;
    }
  }
  if (clusters > p.n_tiles) clusters = p.n_tiles;
  return record_cuda(launch_clusters(kernel, clusters, csize, threads, L.total, stream, tm_h, tm_w, p));
}

// ---------------------------------------------------------------------------
// W1' = W1 diag(w_ln): folds the RMSNorm weight into the first score layer, so the fused
// kernel only has to scale each row's accumulator by its 1 / rms.
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(256) fold_rmsnorm_weight_kernel(const uint16_t *W1, const uint16_t *ln_w,
                                                                  int32_t d_g, int32_t d, uint16_t *W1_out) {
  tg::pdl_wait();
  tg::pdl_launch_dependents();
  const long long n = static_cast<long long>(d_g) * d;
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < n; i += static_cast<long long>(gridDim.x) * 256) {
    const int c = static_cast<int>(i % d);
    W1_out[i] = tg::float_to_bf16_bits(tg::bf16_bits_to_float(W1[i]) * tg::bf16_bits_to_float(ln_w[c]));
  }
}

tg_status launch_fold_rmsnorm_weight(const uint16_t *W1, const uint16_t *ln_w, int32_t d_g, int32_t d,
                                     uint16_t *W1_out, cudaStream_t stream) {
  const long long n = static_cast<long long>(d_g) * d;
  long long grid = (n + 255) / 256;
  if (grid > num_sms() * 8) grid = num_sms() * 8;
  return record_cuda(launch_pdl(fold_rmsnorm_weight_kernel, dim3(static_cast<int>(grid)), dim3(256), 0, stream,
                                W1, ln_w, d_g, d, W1_out));
}

}  // namespace tg_host
