// tg_select.cu — top-K selection and keep-index compaction (TokenGate deep dive, section
// 3.1, Eq. (4): S = topK_{j in P}(b_j) union N; section 3.4: budget clamped to |P|, keep
// indices over the full sequence in original order).
//
// One thread-block cluster of kCluster CTAs per sequence; CTA r owns the r-th contiguous
// chunk of the sequence and loads it once into shared memory as order-preserving uint32
// keys (instruction rows -> 0, never selected as documents; NaN -> 1, below every number;
// -0.0 -> +0.0). The K_b-th largest document key is found by an MSB-first radix select in
// three passes of 11, 11 and 10 bits: each CTA builds a 2048-bin histogram of its chunk in
// shared memory with shared atomics and sums it into 64 coarse bins of 32; after a cluster
// barrier every CTA reads the eight coarse histograms through distributed shared memory,
// picks the coarse bin holding the wanted rank, then reads only that coarse bin's 32 fine
// bins from the eight CTAs (two small remote rounds instead of pulling whole histograms,
// since DSMEM bandwidth, not latency, dominated), and every CTA picks the same digit. After the
// third pass the threshold key T and the number of ties at T to keep are exact; ties are
// granted to the lowest indices. When, after the first or second pass, the chosen bin holds
// exactly as many keys as are still needed (the usual case for continuous scores after 22
// bits), the whole bin is kept: T is set just below the bin with no ties to split, and the
// remaining passes are skipped. The kept set is the same either way. Compaction: each warp owns a contiguous segment of its
// CTA's chunk; per-warp counts of keys above / at T and of instruction rows, one DSMEM
// exchange of CTA totals, and one ballot-prefix pass per warp write the kept indices in
// order. No global scratch memory and no waits between clusters: the output offset of
// sequence b is rebuilt by each cluster from the instruction-token counts before it.
#include <cooperative_groups.h>

#include "tg_common.cuh"

namespace cg = cooperative_groups;

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kCluster = 8;
constexpr int kMaxB = 1024;
constexpr int kBins = 2048;  // 11-bit digits
constexpr int kFine = 32;    // fine bins per coarse bin
constexpr int kCoarse = kBins / kFine;
constexpr int kMaxSmemKeys = 40960;  // 160 KB; longer chunks stream their keys from L2
static_assert(kBins == 4 * kThreads, "each thread owns four histogram bins");
static_assert(kCoarse * kCluster == kThreads, "one thread per (coarse bin, rank)");

struct SelectParams {
  const float *s;
  const uint8_t *mask;
  const int32_t *cu_seqlens;
  int32_t B, T, K, capacity, smem_keys;
  int32_t cu_base;  // added to every cu_kept value (a list packed after cu_base earlier rows)
  int32_t vec;  // s is 16-byte and mask 4-byte aligned: stage keys with vector loads
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

// Cluster barrier halves: arrive publishes this thread's earlier shared-memory writes to
// the cluster, wait makes every other CTA's writes before its arrive visible here.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  cluster_arrive();
  cluster_wait();
}

// Load a 32-bit word from the shared memory of CTA `rank` of this cluster.
__device__ __forceinline__ int32_t ld_peer(const int32_t *local_addr, int rank) {
  uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local_addr)), r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  int32_t v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(r) : "memory");
  return v;
}
__device__ __forceinline__ int4 ld_peer4(const int4 *local_addr, int rank) {
  uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local_addr)), r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  int4 v;
  asm volatile("ld.shared::cluster.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(r)
               : "memory");
  return v;
}

// Sum over the 8 consecutive lanes of a lane group (lane & ~7 .. lane | 7).
__device__ __forceinline__ int sum8(int v) {
  v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
  v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
  v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
  return v;
}

// Inclusive suffix sum over the lanes of a warp (lane l gets the sum of lanes l..31).
__device__ __forceinline__ int warp_suffix(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_down_sync(0xFFFFFFFFu, v, o);
    if (lane + o < 32) v += t;
  }
  return v;
}

struct SelShared {
  int32_t hist[2][kBins];     // fine histogram, double-buffered by pass parity
  int32_t coarse[2][kCoarse]; // sums of 32 consecutive fine bins, same buffering
  int32_t ctot[kCoarse];      // cluster-wide coarse totals
  int32_t ftot[kFine];        // cluster-wide counts of the fine bins inside the chosen coarse bin
  int32_t pick[3][5];         // per pass: coarse bin, keys needed in it, digit, keys needed in it,
                              // keys in that digit's bin
  int32_t n_need;             // keys the selection takes: min(K, document rows)
  int32_t wgt[kWarps], weq[kWarps], wnm[kWarps];
  int32_t woff[kWarps], wtie[kWarps];
  int32_t red[kWarps];
  int4 xch;                 // this CTA's counts: keys > T, keys == T, instruction rows
  int32_t m_b;              // the sequence's end offset in the kept list
  int32_t prev_cnt[kMaxB];  // instruction rows of each earlier sequence inside this chunk
  int32_t cus[kMaxB + 1];   // cu_seqlens of the earlier sequences (for the searches of that count)
};

// Block-wide sum of one int per thread (valid in every thread).
__device__ __forceinline__ int block_sum(int v, SelShared &sh) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  if (lane == 0) sh.red[warp] = v;
  __syncthreads();
  int r = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) r += sh.red[w];
  __syncthreads();
  return r;
}

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, 1)
    topk_select_kernel(SelectParams p) {
  __shared__ __align__(16) SelShared sh;
  extern __shared__ uint32_t ks[];
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int b = blockIdx.x / kCluster;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  tg::pdl_wait();
  tg::pdl_launch_dependents();

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
  if (in_smem && p.vec) {
    // aligned body with 16-byte score / 4-byte mask loads, scalar head and tail
    const int e = lo + len;
    const int a4 = min(e, (lo + 3) & ~3);
    const int e4 = max(a4, e & ~3);
    for (int j = lo + tid; j < a4; j += kThreads) ks[j - lo] = load_key(p, j);
    for (int j = e4 + tid; j < e; j += kThreads) ks[j - lo] = load_key(p, j);
    const int nv = (e4 - a4) >> 2;
    const float4 *s4 = reinterpret_cast<const float4 *>(p.s + a4);
    const uchar4 *m4 = reinterpret_cast<const uchar4 *>(p.mask + a4);
    uint32_t *dst = ks + (a4 - lo);
    for (int v = tid; v < nv; v += 2 * kThreads) {
      const bool two = v + kThreads < nv;
      const float4 x0 = s4[v];
      const float4 x1 = two ? s4[v + kThreads] : x0;
      const uchar4 q0 = p.mask ? m4[v] : make_uchar4(0, 0, 0, 0);
      const uchar4 q1 = (p.mask && two) ? m4[v + kThreads] : make_uchar4(0, 0, 0, 0);
      dst[4 * v + 0] = q0.x ? 0u : order_key(x0.x);
      dst[4 * v + 1] = q0.y ? 0u : order_key(x0.y);
      dst[4 * v + 2] = q0.z ? 0u : order_key(x0.z);
      dst[4 * v + 3] = q0.w ? 0u : order_key(x0.w);
      if (two) {
        uint32_t *d1 = dst + 4 * (v + kThreads);
        d1[0] = q1.x ? 0u : order_key(x1.x);
        d1[1] = q1.y ? 0u : order_key(x1.y);
        d1[2] = q1.z ? 0u : order_key(x1.z);
        d1[3] = q1.w ? 0u : order_key(x1.w);
      }
    }
  } else if (in_smem) {
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
    for (int i = tid; i <= b; i += kThreads) sh.cus[i] = p.cu_seqlens[i];
    __syncthreads();
    // largest sequence index in [0, b) starting at or before row j
    auto count_row = [&](int j) {
      int lo_b = 0, hi_b = b;
      while (hi_b - lo_b > 1) {
        const int mid = (lo_b + hi_b) >> 1;
        if (sh.cus[mid] <= j) lo_b = mid; else hi_b = mid;
      }
      atomicAdd(&sh.prev_cnt[lo_b], 1);
    };
    const int share = (start + kCluster - 1) / kCluster;
    const int a0 = min(start, rank * share), a1 = min(start, (rank + 1) * share);
    // whole 4-byte words of the mask in [w0, w1) (mask is 4-byte aligned when p.vec), four words
    // in flight per thread; the bytes before and after them one at a time
    const int w0 = p.vec ? min(a1, (a0 + 3) & ~3) : a1;
    const int w1 = p.vec ? max(w0, a1 & ~3) : a1;
    for (int j = a0 + tid; j < w0; j += kThreads)
      if (p.mask[j]) count_row(j);
    for (int j = w1 + tid; j < a1; j += kThreads)
      if (p.mask[j]) count_row(j);
    const uchar4 *m4 = reinterpret_cast<const uchar4 *>(p.mask);
    const int v0 = w0 >> 2, v1 = w1 >> 2;
    int v = v0 + tid;
    for (; v + 3 * kThreads < v1; v += 4 * kThreads) {
      uchar4 q[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) q[u] = m4[v + u * kThreads];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = 4 * (v + u * kThreads);
        if (q[u].x) count_row(j);
        if (q[u].y) count_row(j + 1);
        if (q[u].z) count_row(j + 2);
        if (q[u].w) count_row(j + 3);
      }
    }
    for (; v < v1; v += kThreads) {
      const uchar4 q = m4[v];
      const int j = 4 * v;
      if (q.x) count_row(j);
      if (q.y) count_row(j + 1);
      if (q.z) count_row(j + 2);
      if (q.w) count_row(j + 3);
    }
  }

  // ---- radix select: 11 + 11 + 10 bits, MSB first ----
  uint32_t prefix = 0;
  int need = 0;
  int seq_offset = 0;
  bool select_none = false;
  bool early = false;
  uint32_t early_t = 0u;
  for (int pass = 0; pass < 3; ++pass) {
    int32_t *hist = sh.hist[pass & 1];
    reinterpret_cast<int4 *>(hist)[tid] = make_int4(0, 0, 0, 0);
    __syncthreads();
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int width = pass < 2 ? 11 : 10;
    const uint32_t dmask = (1u << width) - 1u;
    // four keys in flight per thread: the shared-memory loads go out before the atomics
    int i = tid;
    for (; i + 3 * kThreads < len; i += 4 * kThreads) {
      uint32_t k4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) k4[u] = key_at(i + u * kThreads);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (k4[u] != 0u && (pass == 0 || (k4[u] >> (shift + width)) == prefix))
          atomicAdd(&hist[(k4[u] >> shift) & dmask], 1);
    }
    for (; i < len; i += kThreads) {
      const uint32_t key = key_at(i);
      if (key != 0u && (pass == 0 || (key >> (shift + width)) == prefix))
        atomicAdd(&hist[(key >> shift) & dmask], 1);
    }
    __syncthreads();
    {
      // local coarse histogram: thread t sums fine bins 4t..4t+3; 8 lanes make a coarse bin
      const int4 f = reinterpret_cast<const int4 *>(hist)[tid];
      const int c8 = sum8(f.x + f.y + f.z + f.w);
      if ((lane & 7) == 0) sh.coarse[pass & 1][tid >> 3] = c8;
    }
    cluster_sync_all();
    if (pass == 0 && b > 0) {
      // earlier sequences: sum of min(n_i, K + |N_i|) = sum of (K_i + |N_i|)
      int part = 0;
      for (int i = tid; i < b; i += kThreads) {
        int c = 0;
        for (int r = 0; r < kCluster; ++r) c += ld_peer(&sh.prev_cnt[i], r);
        part += min(p.cu_seqlens[i + 1] - p.cu_seqlens[i], p.K + c);
      }
      seq_offset = block_sum(part, sh);
    }
    // round 1: cluster-wide coarse totals; thread t reads coarse bin t/8 of rank t%8
    {
      const int ct = sum8(ld_peer(&sh.coarse[pass & 1][tid >> 3], tid & 7));
      if ((lane & 7) == 0) sh.ctot[tid >> 3] = ct;
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns coarse bins 2l and 2l+1; find the one holding the need-th largest key
      const int lo_c = sh.ctot[2 * lane], hi_c = sh.ctot[2 * lane + 1];
      const int suf = warp_suffix(lo_c + hi_c);
      const int all = __shfl_sync(0xFFFFFFFFu, suf, 0);
      const int nd = pass == 0 ? min(p.K, all) : need;
      if (lane == 0 && pass == 0) sh.n_need = nd;
      const int above = suf - lo_c - hi_c;
      if (above < nd && nd <= above + hi_c) {
        sh.pick[pass][0] = 2 * lane + 1;
        sh.pick[pass][1] = nd - above;
      } else if (above + hi_c < nd && nd <= above + hi_c + lo_c) {
        sh.pick[pass][0] = 2 * lane;
        sh.pick[pass][1] = nd - above - hi_c;
      }
    }
    __syncthreads();
    if (pass == 0) {
      need = sh.n_need;
      if (need == 0) {
        select_none = true;
        break;  // uniform: every CTA of the cluster sees the same count
      }
    }
    // round 2: cluster-wide counts of the 32 fine bins inside the chosen coarse bin
    const int cbin = sh.pick[pass][0];
    if (tid < kFine * kCluster) {
      const int ft = sum8(ld_peer(&hist[cbin * kFine + (tid >> 3)], tid & 7));
      if ((lane & 7) == 0) sh.ftot[tid >> 3] = ft;
    }
    __syncthreads();
    if (warp == 0) {
      const int nd = sh.pick[pass][1];
      const int cnt = sh.ftot[lane];
      const int above = warp_suffix(cnt) - cnt;
      if (above < nd && nd <= above + cnt) {
        sh.pick[pass][2] = cbin * kFine + lane;
        sh.pick[pass][3] = nd - above;
        sh.pick[pass][4] = cnt;
      }
    }
    __syncthreads();
    prefix = (prefix << width) | static_cast<uint32_t>(sh.pick[pass][2]);
    need = sh.pick[pass][3];
    if (pass < 2 && need == sh.pick[pass][4] && prefix != 0u) {
      // every key of the chosen bin is kept: the threshold sits just below the bin, with no
      // ties to split, and the remaining passes are not needed (uniform: every CTA of the
      // cluster read the same counts)
      early_t = (prefix << shift) - 1u;
      early = true;
      break;
    }
  }
  const uint32_t T = select_none ? 0xFFFFFFFFu : (early ? early_t : prefix);
  const int need_ties = (select_none || early) ? 0 : need;

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
    int g = lane < kWarps ? sh.wgt[lane] : 0;
    int e = lane < kWarps ? sh.weq[lane] : 0;
    int m = lane < kWarps ? sh.wnm[lane] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      g += __shfl_xor_sync(0xFFFFFFFFu, g, o);
      e += __shfl_xor_sync(0xFFFFFFFFu, e, o);
      m += __shfl_xor_sync(0xFFFFFFFFu, m, o);
    }
    if (lane == 0) sh.xch = make_int4(g, e, m, 0);
  }
  cluster_sync_all();
  if (warp == 0) {
    // lane r < kCluster holds rank r's counts; prefix over ranks in rank (= index) order
    const int4 x = lane < kCluster ? ld_peer4(&sh.xch, lane) : make_int4(0, 0, 0, 0);
    int eq_incl = x.y;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, eq_incl, o);
      if (lane >= o) eq_incl += t;
    }
    const int eq_excl = eq_incl - x.y;
    const int ties_r = max(0, min(need_ties - eq_excl, x.y));
    const int keep_r = x.x + ties_r + x.z;
    int keep_incl = keep_r;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, keep_incl, o);
      if (lane >= o) keep_incl += t;
    }
    const int eq_before = __shfl_sync(0xFFFFFFFFu, eq_excl, rank);
    const int keep_before = __shfl_sync(0xFFFFFFFFu, keep_incl - keep_r, rank);
    const int M_b = __shfl_sync(0xFFFFFFFFu, keep_incl, kCluster - 1);
    if (lane == 0) sh.m_b = seq_offset + M_b;
    // per-warp tie base and output offset, in warp (= index) order
    const int e = lane < kWarps ? sh.weq[lane] : 0;
    int e_incl = e;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, e_incl, o);
      if (lane >= o) e_incl += t;
    }
    const int tie_base = eq_before + e_incl - e;
    const int ties_w = max(0, min(need_ties - tie_base, e));
    const int keep_w = lane < kWarps ? sh.wgt[lane] + sh.wnm[lane] + ties_w : 0;
    int k_incl = keep_w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, k_incl, o);
      if (lane >= o) k_incl += t;
    }
    if (lane < kWarps) {
      sh.wtie[lane] = tie_base;
      sh.woff[lane] = seq_offset + keep_before + k_incl - keep_w;
    }
  }
  __syncthreads();
  // this CTA is done reading its peers' shared memory (the loads have returned)
  cluster_arrive_relaxed();
  if (rank == 0 && tid == 0) {
    if (b == 0) p.cu_kept[0] = p.cu_base;
    p.cu_kept[b + 1] = p.cu_base + sh.m_b;
  }

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
  cluster_wait();
}

}  // namespace

namespace tg_host {

tg_status launch_topk_select(const float *s, const uint8_t *mask, const int32_t *cu_seqlens,
                             int32_t B, int32_t T, int32_t K, int32_t *kept_idx, int32_t capacity,
                             int32_t *cu_kept, int32_t *status, cudaStream_t stream, int32_t cu_base) {
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
  p.cu_base = cu_base;
  // every sequence is at most T long, so its chunk is at most ceil(T / kCluster) keys
  int keys = (T + kCluster - 1) / kCluster;
  keys = keys < 1 ? 1 : (keys > kMaxSmemKeys ? kMaxSmemKeys : keys);
  p.smem_keys = keys;
  p.vec = (reinterpret_cast<uintptr_t>(s) % 16 == 0) &&
          (mask == nullptr || reinterpret_cast<uintptr_t>(mask) % 4 == 0);
  const size_t smem = static_cast<size_t>(keys) * 4;
  cudaError_t e = cudaFuncSetAttribute(topk_select_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return record_cuda(e);
  return record_cuda(launch_pdl(topk_select_kernel, dim3(B * kCluster), dim3(kThreads), smem, stream, p));
}

}  // namespace tg_host
