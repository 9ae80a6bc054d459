// tg_select.cu — top-K selection and keep-index compaction (TokenGate deep dive, section
// 3.1, Eq. (4): S = topK_{j in P}(b_j) union N; section 3.4: budget clamped to |P|, keep
// indices over the full sequence in original order).
//
// One thread-block cluster of kCluster CTAs per sequence; CTA r of the cluster owns the
// r-th contiguous chunk of the sequence. Scores are mapped to order-preserving uint32 keys
// (NaN -> 0, below every number; -0.0 -> +0.0) and the K_b-th largest key is found by an
// MSB-first radix select, 8 bits per pass: each CTA builds a 256-bin histogram of its
// chunk in shared memory with warp-aggregated atomics (__match_any_sync), the cluster sums
// the eight histograms through distributed shared memory, and every CTA picks the same
// bin. After four passes the threshold key T and the number of ties at T to keep are
// exact. Ties are then granted to the lowest indices: each CTA learns how many ties and
// kept rows lie in the chunks before it (one DSMEM exchange of three counts) and writes
// its kept indices in order with ballot-based block scans. No global scratch memory, no
// inter-cluster waits: the output offset of sequence b is recomputed by each cluster from
// the instruction-token counts of the sequences before it.
#include <cooperative_groups.h>

#include "tg_common.cuh"

namespace cg = cooperative_groups;

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kCluster = 8;
constexpr int kMaxB = 1024;

struct SelectParams {
  const float *s;
  const uint8_t *mask;
  const int32_t *cu_seqlens;
  int32_t B, T, K, capacity;
  int32_t *kept_idx;
  int32_t *cu_kept;
  int32_t *status;
};

__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0u;  // NaN ranks below every number
  if (u == 0x80000000u) u = 0u;                      // -0.0 ties with +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct SelShared {
  int32_t hist[2][256];
  int32_t warp_tot[kWarps];
  int32_t scan_tmp[kWarps];
  int32_t xch[4];        // this CTA's counts: [0] keys > T, [1] keys == T, [2] instr rows
  int32_t bcast[4];      // block broadcast slots
  int32_t prev_cnt[kMaxB];  // instruction-token counts of earlier sequences (this CTA's part)
};

// Block-wide exclusive scan of one 0/1 flag per thread; returns the prefix, *total = sum.
__device__ __forceinline__ int block_excl_scan_flag(bool flag, SelShared &sh, int *total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned bal = __ballot_sync(0xFFFFFFFFu, flag);
  const int in_warp = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) sh.warp_tot[warp] = __popc(bal);
  __syncthreads();
  if (warp == 0) {
    int v = sh.warp_tot[lane];
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += t;
    }
    sh.scan_tmp[lane] = incl - v;
    if (lane == 31) sh.bcast[3] = incl;
  }
  __syncthreads();
  const int r = sh.scan_tmp[warp] + in_warp;
  *total = sh.bcast[3];
  __syncthreads();
  return r;
}

// Block-wide sum of one int per thread (result valid in every thread).
__device__ __forceinline__ int block_sum(int v, SelShared &sh) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  if (lane == 0) sh.warp_tot[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int x = sh.warp_tot[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
    if (lane == 0) sh.bcast[2] = x;
  }
  __syncthreads();
  const int r = sh.bcast[2];
  __syncthreads();
  return r;
}

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, 1)
    topk_select_kernel(SelectParams p) {
  __shared__ SelShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int b = blockIdx.x / kCluster;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  // ---- validate this sequence's bounds (uniform across the cluster) ----
  const int start = p.cu_seqlens[b];
  const int end = p.cu_seqlens[b + 1];
  const bool bad = start < 0 || end < start || end > p.T ||
                   (b == 0 && start != 0) || (b == p.B - 1 && end != p.T);
  if (bad) {
    if (rank == 0 && tid == 0) tg::report(p.status, TG_DEV_BAD_SEQLENS);
    return;
  }
  const int n = end - start;
  const int chunk = (n + kCluster - 1) / kCluster;
  const int lo = start + min(n, rank * chunk);
  const int hi = start + min(n, (rank + 1) * chunk);

  // ---- output offset of this sequence: sum over earlier sequences of min(n_b', K + |N_b'|) ----
  for (int i = tid; i < b; i += kThreads) sh.prev_cnt[i] = 0;
  __syncthreads();
  if (p.mask != nullptr && b > 0) {
    // this CTA counts instruction tokens in its 1/kCluster share of rows [0, start)
    const int share = (start + kCluster - 1) / kCluster;
    const int a0 = min(start, rank * share), a1 = min(start, (rank + 1) * share);
    int cur = 0;  // sequence of the row being scanned (rows visited in increasing order)
    for (int j = a0 + tid; j < a1; j += kThreads) {
      if (p.mask[j]) {
        // binary search the sequence holding row j
        int lo_b = 0, hi_b = b;  // answer in [0, b)
        while (hi_b - lo_b > 1) {
          const int mid = (lo_b + hi_b) >> 1;
          if (p.cu_seqlens[mid] <= j) lo_b = mid; else hi_b = mid;
        }
        cur = lo_b;
        atomicAdd(&sh.prev_cnt[cur], 1);
      }
    }
  }
  cluster.sync();
  int my_offset_part = 0;
  for (int i = tid; i < b; i += kThreads) {
    int c = 0;
    for (int r = 0; r < kCluster; ++r) c += cluster.map_shared_rank(&sh, r)->prev_cnt[i];
    const int n_i = p.cu_seqlens[i + 1] - p.cu_seqlens[i];
    my_offset_part += min(n_i, p.K + c);  // = min(K, |P_i|) + |N_i|
  }
  const int seq_offset = block_sum(my_offset_part, sh);

  // ---- radix select: 4 passes of 8 bits, MSB first ----
  uint32_t prefix = 0;
  int need = 0;          // how many keys to take among those matching `prefix`
  int K_b = 0;
  int n_doc = 0;
  bool select_none = false;
  for (int pass = 0; pass < 4; ++pass) {
    int32_t *hist = sh.hist[pass & 1];
    if (tid < 256) hist[tid] = 0;
    __syncthreads();
    const int shift = 24 - 8 * pass;
    for (int base = lo; base < hi; base += kThreads) {
      const int j = base + tid;
      int bin = -1;
      if (j < hi && !(p.mask && p.mask[j])) {
        const uint32_t key = order_key(p.s[j]);
        if (pass == 0 || (key >> (shift + 8)) == prefix) bin = static_cast<int>((key >> shift) & 255u);
      }
      const unsigned peers = __match_any_sync(0xFFFFFFFFu, bin);
      if (bin >= 0 && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
    }
    cluster.sync();
    // cluster-wide histogram; thread t owns bin 255 - t so an inclusive scan over t gives
    // the number of keys in bins >= 255 - t
    int tot = 0, bin_id = 255 - tid;
    if (tid < 256)
      for (int r = 0; r < kCluster; ++r) tot += cluster.map_shared_rank(hist, r)[bin_id];
    if (pass == 0) {
      n_doc = block_sum(tid < 256 ? tot : 0, sh);
      K_b = min(p.K, n_doc);
      need = K_b;
      if (K_b == 0) {
        select_none = true;
        break;  // uniform: every CTA of the cluster computed the same K_b
      }
    }
    // inclusive scan over the 256 bins (warps 0-7)
    int incl = tot;
    if (tid < 256) {
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
      }
      if (lane == 31) sh.scan_tmp[warp] = incl;
    }
    __syncthreads();
    if (tid < 256) {
      int add = 0;
      for (int w = 0; w < warp; ++w) add += sh.scan_tmp[w];
      incl += add;
      const int above = incl - tot;
      if (above < need && need <= incl) {
        sh.bcast[0] = bin_id;
        sh.bcast[1] = need - above;
      }
    }
    __syncthreads();
    prefix = (prefix << 8) | static_cast<uint32_t>(sh.bcast[0]);
    need = sh.bcast[1];
    __syncthreads();
  }
  const uint32_t T = select_none ? 0xFFFFFFFFu : prefix;
  const int need_ties = select_none ? 0 : need;

  // ---- per-CTA counts of keys above / at the threshold and of instruction rows ----
  int c_gt = 0, c_eq = 0, c_nm = 0;
  for (int j = lo + tid; j < hi; j += kThreads) {
    if (p.mask && p.mask[j]) {
      ++c_nm;
    } else {
      const uint32_t key = order_key(p.s[j]);
      c_gt += key > T;
      c_eq += key == T;
    }
  }
  c_gt = block_sum(c_gt, sh);
  c_eq = block_sum(c_eq, sh);
  c_nm = block_sum(c_nm, sh);
  if (tid == 0) {
    sh.xch[0] = c_gt;
    sh.xch[1] = c_eq;
    sh.xch[2] = c_nm;
  }
  cluster.sync();
  int eq_before = 0, keep_before = 0, M_b = 0;
  {
    int eq_run = 0;
    for (int r = 0; r < kCluster; ++r) {
      const int32_t *x = cluster.map_shared_rank(sh.xch, r);
      const int ties_r = max(0, min(need_ties - eq_run, x[1]));
      const int keep_r = x[0] + ties_r + x[2];
      if (r < rank) {
        eq_before += x[1];
        keep_before += keep_r;
      }
      eq_run += x[1];
      M_b += keep_r;
    }
  }
  if (rank == 0 && tid == 0) {
    if (b == 0) p.cu_kept[0] = 0;
    p.cu_kept[b + 1] = seq_offset + M_b;
  }

  // ---- order-preserving compaction of this CTA's chunk ----
  int run_ties = eq_before;
  int run_keep = seq_offset + keep_before;
  bool overflow = false;
  for (int base = lo; base < hi; base += kThreads) {
    const int j = base + tid;
    const bool valid = j < hi;
    const bool instr = valid && p.mask && p.mask[j];
    uint32_t key = 0;
    if (valid && !instr) key = order_key(p.s[j]);
    const bool is_doc = valid && !instr;
    const bool tie = is_doc && key == T;
    int tile_ties;
    const int tie_rank = run_ties + block_excl_scan_flag(tie, sh, &tile_ties);
    const bool keep = instr || (is_doc && key > T) || (tie && tie_rank < need_ties);
    int tile_keep;
    const int out = run_keep + block_excl_scan_flag(keep, sh, &tile_keep);
    if (keep) {
      if (out >= 0 && out < p.capacity) p.kept_idx[out] = j;
      else overflow = true;
    }
    run_ties += tile_ties;
    run_keep += tile_keep;
  }
  if (overflow) tg::report(p.status, TG_DEV_CAPACITY);
  // keep this CTA's shared memory alive until every peer has finished reading it
  cluster.sync();
}

}  // namespace

namespace tg_host {

tg_status launch_topk_select(const float *s, const uint8_t *mask, const int32_t *cu_seqlens,
                             int32_t B, int32_t T, int32_t K, int32_t *kept_idx, int32_t capacity,
                             int32_t *cu_kept, int32_t *status, cudaStream_t stream) {
  SelectParams p;
  p.s = s;
  p.mask = mask;
  p.cu_seqlens = cu_seqlens;
  p.B = B;
  p.T = T;
  p.K = K;
  p.capacity = capacity;
  p.kept_idx = kept_idx;
  p.cu_kept = cu_kept;
  p.status = status;
  topk_select_kernel<<<B * kCluster, kThreads, 0, stream>>>(p);
  return record_cuda(cudaGetLastError());
}

}  // namespace tg_host
