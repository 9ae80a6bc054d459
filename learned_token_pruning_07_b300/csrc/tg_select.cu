// tg_select.cu — top-K selection and keep-index compaction (TokenGate deep dive, section
// 3.1, Eq. (4): S = topK_{j in P}(b_j) union N; section 3.4: budget clamped to |P|, keep
// indices over the full sequence in original order).
//
// One thread-block cluster of kCluster CTAs per sequence; CTA r owns the r-th contiguous
// chunk of the sequence and loads it once into shared memory as order-preserving uint32
// keys (instruction rows -> 0, never selected as documents; NaN -> 1, below every number;
// -0.0 -> +0.0). The K_b-th largest document key is found by an MSB-first radix select in
// three passes of 11, 11 and 10 bits: each CTA builds a 2048-bin histogram of its chunk in
// shared memory with warp-aggregated atomics (__match_any_sync), the cluster sums the eight
// histograms through distributed shared memory, and every CTA picks the same bin. After the
// third pass the threshold key T and the number of ties at T to keep are exact; ties are
// granted to the lowest indices. Compaction: each warp owns a contiguous segment of its
// CTA's chunk; per-warp counts of keys above / at T and of instruction rows, one DSMEM
// exchange of CTA totals, and one ballot-prefix pass per warp write the kept indices in
// order. No global scratch memory and no waits between clusters: the output offset of
// sequence b is rebuilt by each cluster from the instruction-token counts before it.
#include <cooperative_groups.h>

#include "tg_common.cuh"

namespace cg = cooperative_groups;

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kCluster = 8;
constexpr int kMaxB = 1024;
constexpr int kBins = 2048;
constexpr int kMaxSmemKeys = 40960;  // 160 KB; longer chunks stream their keys from L2

struct SelectParams {
  const float *s;
  const uint8_t *mask;
  const int32_t *cu_seqlens;
  int32_t B, T, K, capacity, smem_keys;
  int32_t *kept_idx;
  int32_t *cu_kept;
  int32_t *status;
};

// Order-preserving key of a document score; instruction rows get 0.
__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 1u;   // NaN ranks below every number
  if (u == 0x80000000u) u = 0u;                       // -0.0 ties with +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // -inf -> 0x007FFFFF > 1
}

__device__ __forceinline__ uint32_t load_key(const SelectParams &p, int j) {
  const float v = p.s[j];  // both loads issued before either is used
  const uint8_t m = p.mask ? p.mask[j] : uint8_t(0);
  return m ? 0u : order_key(v);
}

struct SelShared {
  int32_t hist[2][kBins];
  int32_t warp_tot[kWarps];
  int32_t wgt[kWarps], weq[kWarps], wnm[kWarps];
  int32_t woff[kWarps], wtie[kWarps];
  int32_t xch[4];  // this CTA's counts: [0] keys > T, [1] keys == T, [2] instruction rows
  int32_t bcast[4];
  int32_t prev_cnt[kMaxB];
};

// Block-wide sum of one int per thread (valid in every thread).
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
  extern __shared__ uint32_t ks[];
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int b = blockIdx.x / kCluster;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  // ---- this sequence's bounds (uniform across the cluster) ----
  const int start = p.cu_seqlens[b];
  const int end = p.cu_seqlens[b + 1];
  const bool bad = start < 0 || end < start || end > p.T || (b == 0 && start != 0) ||
                   (b == p.B - 1 && end != p.T);
  if (bad) {
    if (rank == 0 && tid == 0) tg::report(p.status, TG_DEV_BAD_SEQLENS);
    return;
  }
  const int n = end - start;
  const int chunk = (n + kCluster - 1) / kCluster;
  const int lo = start + min(n, rank * chunk);
  const int len = min(n, (rank + 1) * chunk) - min(n, rank * chunk);
  const bool in_smem = chunk <= p.smem_keys;
  auto key_at = [&](int i) -> uint32_t { return in_smem ? ks[i] : load_key(p, lo + i); };

  // ---- stage keys in shared memory; count instruction rows of earlier sequences ----
  for (int i = tid; i < b; i += kThreads) sh.prev_cnt[i] = 0;
  if (in_smem) {
    int i = tid;
    for (; i + 3 * kThreads < len; i += 4 * kThreads) {
      const uint32_t k0 = load_key(p, lo + i), k1 = load_key(p, lo + i + kThreads);
      const uint32_t k2 = load_key(p, lo + i + 2 * kThreads), k3 = load_key(p, lo + i + 3 * kThreads);
      ks[i] = k0;
      ks[i + kThreads] = k1;
      ks[i + 2 * kThreads] = k2;
      ks[i + 3 * kThreads] = k3;
    }
    for (; i < len; i += kThreads) ks[i] = load_key(p, lo + i);
  }
  __syncthreads();
  if (p.mask != nullptr && b > 0) {
    const int share = (start + kCluster - 1) / kCluster;
    const int a0 = min(start, rank * share), a1 = min(start, (rank + 1) * share);
    for (int j = a0 + tid; j < a1; j += kThreads) {
      if (p.mask[j]) {
        int lo_b = 0, hi_b = b;  // largest sequence index in [0, b) starting at or before j
        while (hi_b - lo_b > 1) {
          const int mid = (lo_b + hi_b) >> 1;
          if (p.cu_seqlens[mid] <= j) lo_b = mid; else hi_b = mid;
        }
        atomicAdd(&sh.prev_cnt[lo_b], 1);
      }
    }
  }

  // ---- radix select: 11 + 11 + 10 bits, MSB first ----
  uint32_t prefix = 0;
  int need = 0;
  int seq_offset = 0;
  bool select_none = false;
  for (int pass = 0; pass < 3; ++pass) {
    int32_t *hist = sh.hist[pass & 1];
    for (int i = tid; i < kBins; i += kThreads) hist[i] = 0;
    __syncthreads();
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int width = pass < 2 ? 11 : 10;
    const uint32_t dmask = (1u << width) - 1u;
    for (int base = 0; base < len; base += kThreads) {
      const int i = base + tid;
      int bin = -1;
      if (i < len) {
        const uint32_t key = key_at(i);
        if (key != 0u && (pass == 0 || (key >> (shift + width)) == prefix))
          bin = static_cast<int>((key >> shift) & dmask);
      }
      const unsigned peers = __match_any_sync(0xFFFFFFFFu, bin);
      if (bin >= 0 && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
    }
    cluster.sync();
    if (pass == 0) {
      // earlier sequences: sum of min(n_i, K + |N_i|) = sum of (K_i + |N_i|)
      int part = 0;
      for (int i = tid; i < b; i += kThreads) {
        int c = 0;
        for (int r = 0; r < kCluster; ++r) c += cluster.map_shared_rank(&sh, r)->prev_cnt[i];
        part += min(p.cu_seqlens[i + 1] - p.cu_seqlens[i], p.K + c);
      }
      seq_offset = block_sum(part, sh);
    }
    // cluster-wide histogram; thread t owns bins 2047-2t and 2046-2t (descending order)
    const int bin_hi = kBins - 1 - 2 * tid, bin_lo = bin_hi - 1;
    int c_hi = 0, c_lo = 0;
#pragma unroll
    for (int r = 0; r < kCluster; ++r) {
      const int32_t *h = cluster.map_shared_rank(hist, r);
      c_hi += h[bin_hi];
      c_lo += h[bin_lo];
    }
    if (pass == 0) {
      const int n_doc = block_sum(c_hi + c_lo, sh);
      need = min(p.K, n_doc);
      if (need == 0) {
        select_none = true;
        break;  // uniform: every CTA of the cluster sees the same n_doc
      }
    }
    // inclusive scan of (c_hi + c_lo) over threads = keys in bins >= bin_lo
    int incl = c_hi + c_lo;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) sh.warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int v = sh.warp_tot[lane];
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += t;
      }
      sh.wgt[lane] = x - v;  // exclusive prefix of warp totals (scratch)
    }
    __syncthreads();
    incl += sh.wgt[warp];
    const int above_hi = incl - c_hi - c_lo;  // keys in bins > bin_hi
    if (above_hi < need && need <= above_hi + c_hi) {
      sh.bcast[0] = bin_hi;
      sh.bcast[1] = need - above_hi;
    } else if (above_hi + c_hi < need && need <= incl) {
      sh.bcast[0] = bin_lo;
      sh.bcast[1] = need - above_hi - c_hi;
    }
    __syncthreads();
    prefix = (prefix << width) | static_cast<uint32_t>(sh.bcast[0]);
    need = sh.bcast[1];
    __syncthreads();
  }
  const uint32_t T = select_none ? 0xFFFFFFFFu : prefix;
  const int need_ties = select_none ? 0 : need;

  // ---- per-warp counts over contiguous warp segments ----
  const int seg = 32 * ((chunk + kThreads - 1) / kThreads);
  const int w0 = min(len, warp * seg), w1 = min(len, (warp + 1) * seg);
  int c_gt = 0, c_eq = 0, c_nm = 0;
  for (int i = w0 + lane; i < w1; i += 32) {
    const uint32_t key = key_at(i);
    c_nm += key == 0u;
    c_gt += key != 0u && key > T;
    c_eq += key != 0u && key == T;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    c_gt += __shfl_xor_sync(0xFFFFFFFFu, c_gt, o);
    c_eq += __shfl_xor_sync(0xFFFFFFFFu, c_eq, o);
    c_nm += __shfl_xor_sync(0xFFFFFFFFu, c_nm, o);
  }
  if (lane == 0) {
    sh.wgt[warp] = c_gt;
    sh.weq[warp] = c_eq;
    sh.wnm[warp] = c_nm;
  }
  __syncthreads();
  if (warp == 0) {
    int g = sh.wgt[lane], e = sh.weq[lane], m = sh.wnm[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      g += __shfl_xor_sync(0xFFFFFFFFu, g, o);
      e += __shfl_xor_sync(0xFFFFFFFFu, e, o);
      m += __shfl_xor_sync(0xFFFFFFFFu, m, o);
    }
    if (lane == 0) {
      sh.xch[0] = g;
      sh.xch[1] = e;
      sh.xch[2] = m;
    }
  }
  cluster.sync();
  if (warp == 0) {
    int eq_before = 0, keep_before = 0, M_b = 0, eq_run = 0;
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
    if (rank == 0 && lane == 0) {
      if (b == 0) p.cu_kept[0] = 0;
      p.cu_kept[b + 1] = seq_offset + M_b;
    }
    // per-warp tie base and output offset, in warp (= index) order
    const int e = sh.weq[lane];
    int e_incl = e;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, e_incl, o);
      if (lane >= o) e_incl += t;
    }
    const int tie_base = eq_before + e_incl - e;
    const int ties_w = max(0, min(need_ties - tie_base, e));
    const int keep_w = sh.wgt[lane] + sh.wnm[lane] + ties_w;
    int k_incl = keep_w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, k_incl, o);
      if (lane >= o) k_incl += t;
    }
    sh.wtie[lane] = tie_base;
    sh.woff[lane] = seq_offset + keep_before + k_incl - keep_w;
  }
  __syncthreads();

  // ---- ordered write of this warp's kept rows ----
  int tie_run = sh.wtie[warp];
  int out_run = sh.woff[warp];
  bool overflow = false;
  const unsigned lt = (1u << lane) - 1u;
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const bool valid = i < w1;
    const uint32_t key = valid ? key_at(i) : 0u;
    const bool instr = valid && key == 0u;
    const bool doc = valid && key != 0u;
    const bool tie = doc && key == T;
    const unsigned tb = __ballot_sync(0xFFFFFFFFu, tie);
    const bool keep = instr || (doc && key > T) || (tie && tie_run + __popc(tb & lt) < need_ties);
    const unsigned kb = __ballot_sync(0xFFFFFFFFu, keep);
    if (keep) {
      const int out = out_run + __popc(kb & lt);
      if (out >= 0 && out < p.capacity) p.kept_idx[out] = lo + i;
      else overflow = true;
    }
    tie_run += __popc(tb);
    out_run += __popc(kb);
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
  // every sequence is at most T long, so its chunk is at most ceil(T / kCluster) keys
  int keys = (T + kCluster - 1) / kCluster;
  keys = keys < 1 ? 1 : (keys > kMaxSmemKeys ? kMaxSmemKeys : keys);
  p.smem_keys = keys;
  const size_t smem = static_cast<size_t>(keys) * 4;
  cudaError_t e = cudaFuncSetAttribute(topk_select_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return record_cuda(e);
  topk_select_kernel<<<B * kCluster, kThreads, smem, stream>>>(p);
  return record_cuda(cudaGetLastError());
}

}  // namespace tg_host
