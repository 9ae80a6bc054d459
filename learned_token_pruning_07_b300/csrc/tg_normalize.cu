// tg_normalize.cu — sequence-axis RMS normalisation of the gate scores (TokenGate deep dive,
// section 3.1, Eq. (3)): b_j = s_j / sqrt(mean over the sequence's prunable rows of s^2 + eps),
// and b_j = 0 on the non-prunable rows. Per-head scores s [T, H_g] (section 3.4: a per-head
// bias) are normalised head by head, and the row mean of the normalised heads (the uniform
// head aggregation that selection ranks) is written beside them.
//
// One 8-CTA cluster per sequence. Each CTA sums s^2 per head and counts the prunable rows of
// its contiguous chunk in a fixed order (per thread in index order, then a shuffle tree per
// warp, then the warps in order); the cluster adds the eight partial sums in rank order
// through distributed shared memory, so the result does not depend on timing. Then every CTA
// writes the normalised scores of its chunk.
#include <cooperative_groups.h>

#include "tg_common.cuh"

namespace cg = cooperative_groups;

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kCluster = 8;
constexpr int kMaxGateHeads = 16;

struct NormParams {
  const float *s;
  int32_t H_g;
  const uint8_t *mask;
  const int32_t *cu_seqlens;
  int32_t B, T;
  float eps;
  float *b_out;
  float *b_sel;  // H_g > 1: [T] mean over heads of the normalised scores (or NULL)
  int32_t *status;
};

// GHP: gate heads padded to 1, 2, 4, 8 or 16 (heads past H_g are skipped)
template <int GHP>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, 1)
    normalize_scores_kernel(const __grid_constant__ NormParams p) {
  __shared__ float warp_sq[kWarps][GHP];
  __shared__ int32_t warp_n[kWarps];
  __shared__ float cta_sq[GHP];
  __shared__ int32_t cta_n;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int b = blockIdx.x / kCluster;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  tg::pdl_wait();
  tg::pdl_launch_dependents();

  const int start = p.cu_seqlens[b];
  const int end = p.cu_seqlens[b + 1];
  const bool bad = start < 0 || end < start || end > p.T || (b == 0 && start != 0) ||
                   (b == p.B - 1 && end != p.T);
  if (bad) {
    if (rank == 0 && tid == 0) tg::report(p.status, TG_DEV_BAD_SEQLENS);
    return;  // uniform across the cluster: every CTA read the same bounds
  }
  const int n = end - start;
  const int chunk = (n + kCluster - 1) / kCluster;
  const int lo = start + min(n, rank * chunk);
  const int hi = start + min(n, (rank + 1) * chunk);
  const int H = GHP == 1 ? 1 : p.H_g;

  // GHP = 1: thread t walks rows t, t + kThreads, ... GHP > 1: thread t owns head c = t % GHP of rows
  // t / GHP, t / GHP + kRows, ..., so a warp reads contiguous (row, head) elements and every
  // thread keeps the sum of one head. Either way each sum runs over its rows in index order, then
  // a shuffle tree per warp, then the warps in order.
  constexpr int kRows = kThreads / GHP;  // rows per step of the CTA
  constexpr int kU = 4;                  // rows per thread whose loads are issued together
  const int c_own = tid % GHP;           // GHP > 1: this thread's head
  float sq = 0.0f;  // this thread's sum of squares (of its one head)
  int cnt = 0;
  if constexpr (GHP == 1) {
    // kU rows per step with every load issued first, so their round trips overlap
    int j = lo + tid;
    for (; j + (kU - 1) * kThreads < hi; j += kU * kThreads) {
      uint8_t m[kU];
      float v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        m[u] = p.mask != nullptr ? p.mask[j + u * kThreads] : uint8_t(0);
        v[u] = p.s[j + u * kThreads];
      }
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (m[u] == 0) {
          sq = fmaf(v[u], v[u], sq);
          ++cnt;
        }
    }
    for (; j < hi; j += kThreads)
      if (p.mask == nullptr || p.mask[j] == 0) {
        const float v = p.s[j];
        sq = fmaf(v, v, sq);
        ++cnt;
      }
  } else {
    int j = lo + tid / GHP;
    for (; j + (kU - 1) * kRows < hi; j += kU * kRows) {
      uint8_t m[kU];
      float v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int jj = j + u * kRows;
        m[u] = p.mask != nullptr ? p.mask[jj] : uint8_t(0);
        v[u] = c_own < H ? p.s[static_cast<size_t>(jj) * H + c_own] : 0.0f;
      }
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (m[u] == 0) {
          sq = fmaf(v[u], v[u], sq);
          cnt += c_own == 0;
        }
    }
    for (; j < hi; j += kRows)
      if (p.mask == nullptr || p.mask[j] == 0) {
        const float v = c_own < H ? p.s[static_cast<size_t>(j) * H + c_own] : 0.0f;
        sq = fmaf(v, v, sq);
        cnt += c_own == 0;
      }
  }
  if constexpr (GHP == 1) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sq += __shfl_xor_sync(0xFFFFFFFFu, sq, o);
      cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, o);
    }
  } else {
    // lanes of the same head: xor over the lane bits above the head bits
#pragma unroll
    for (int o = 16; o >= GHP; o >>= 1) sq += __shfl_xor_sync(0xFFFFFFFFu, sq, o);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, o);
  }
  if (lane == 0) warp_n[warp] = cnt;
  if (lane < GHP) warp_sq[warp][lane] = sq;
  __syncthreads();
  if (tid < GHP) {
    float t = 0.0f;
    for (int w = 0; w < kWarps; ++w) t += warp_sq[w][tid];
    cta_sq[tid] = t;
  }
  if (tid == 0) {
    int c = 0;
    for (int w = 0; w < kWarps; ++w) c += warp_n[w];
    cta_n = c;
  }
  cluster.sync();
  __shared__ float inv[GHP];
  if (tid < GHP) {
    float total = 0.0f;
    int n_doc = 0;
    for (int r = 0; r < kCluster; ++r) {  // rank order: the same sum in every CTA
      total += *cluster.map_shared_rank(&cta_sq[tid], r);
      n_doc += *cluster.map_shared_rank(&cta_n, r);
    }
    // a sequence without prunable rows has nothing to scale: every b is 0
    inv[tid] = n_doc > 0 ? 1.0f / sqrtf(total / static_cast<float>(n_doc) + p.eps) : 0.0f;
  }
  __syncthreads();
  if constexpr (GHP == 1) {
    int jw = lo + tid;
    for (; jw + (kU - 1) * kThreads < hi; jw += kU * kThreads) {
      uint8_t m[kU];
      float v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        m[u] = p.mask != nullptr ? p.mask[jw + u * kThreads] : uint8_t(0);
        v[u] = p.s[jw + u * kThreads];
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) p.b_out[jw + u * kThreads] = m[u] != 0 ? 0.0f : v[u] * inv[0];
    }
    for (; jw < hi; jw += kThreads) {
      const bool keep_always = p.mask != nullptr && p.mask[jw] != 0;
      p.b_out[jw] = keep_always ? 0.0f : p.s[jw] * inv[0];
    }
  } else {
    // the GHP consecutive lanes of a row also form its head mean (a shuffle tree over them); every
    // lane of a warp runs the same number of steps, since the shuffles are warp-wide, and rows past
    // the chunk are skipped inside; kU rows per step with their loads issued first
    const float inv_c = c_own < H ? inv[c_own] : 0.0f;
    const int j_first = lo + tid / GHP;
    const int steps = (hi - lo + kRows - 1) / kRows;
    for (int k = 0; k < steps; k += kU) {
      uint8_t m[kU];
      float sv[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int jj = j_first + (k + u) * kRows;
        const bool in = k + u < steps && jj < hi;
        m[u] = (in && p.mask != nullptr) ? p.mask[jj] : uint8_t(0);
        sv[u] = (in && c_own < H) ? p.s[static_cast<size_t>(jj) * H + c_own] : 0.0f;
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        if (k + u >= steps) break;  // uniform across the CTA
        const int jj = j_first + (k + u) * kRows;
        const bool in = jj < hi;
        const float v = m[u] != 0 ? 0.0f : sv[u] * inv_c;
        if (in && c_own < H) p.b_out[static_cast<size_t>(jj) * H + c_own] = v;
        float sum = v;
#pragma unroll
        for (int o = 1; o < GHP; o <<= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
        if (in && p.b_sel != nullptr && c_own == 0) p.b_sel[jj] = sum / static_cast<float>(H);
      }
    }
  }
  cluster.sync();  // keep this CTA's shared memory alive until every peer has read it
}

}  // namespace

namespace tg_host {

tg_status launch_normalize_scores(const float *s, int32_t H_g, const uint8_t *mask, const int32_t *cu_seqlens,
                                  int32_t B, int32_t T, float eps, float *b_out, float *b_sel, int32_t *status,
                                  cudaStream_t stream) {
  if (H_g < 1 || H_g > kMaxGateHeads) return TG_ERR_UNSUPPORTED;
  NormParams p{s, H_g, mask, cu_seqlens, B, T, eps, b_out, b_sel, status};
  const dim3 grid(B * kCluster), block(kThreads);
  switch (H_g == 1 ? 1 : H_g <= 2 ? 2 : H_g <= 4 ? 4 : H_g <= 8 ? 8 : 16) {
    case 1: return record_cuda(launch_pdl(normalize_scores_kernel<1>, grid, block, 0, stream, p));
    case 2: return record_cuda(launch_pdl(normalize_scores_kernel<2>, grid, block, 0, stream, p));
    case 4: return record_cuda(launch_pdl(normalize_scores_kernel<4>, grid, block, 0, stream, p));
    case 8: return record_cuda(launch_pdl(normalize_scores_kernel<8>, grid, block, 0, stream, p));
    default: return record_cuda(launch_pdl(normalize_scores_kernel<16>, grid, block, 0, stream, p));
  }
}

}  // namespace tg_host
