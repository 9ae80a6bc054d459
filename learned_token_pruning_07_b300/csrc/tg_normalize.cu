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

  float sq[GHP];
#pragma unroll
  for (int c = 0; c < GHP; ++c) sq[c] = 0.0f;
  int cnt = 0;
  for (int j = lo + tid; j < hi; j += kThreads) {
    if (p.mask == nullptr || p.mask[j] == 0) {
#pragma unroll
      for (int c = 0; c < GHP; ++c) {
        if (c < H) {
          const float v = p.s[static_cast<size_t>(j) * H + c];
          sq[c] = fmaf(v, v, sq[c]);
        }
      }
      ++cnt;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
    for (int c = 0; c < GHP; ++c) sq[c] += __shfl_xor_sync(0xFFFFFFFFu, sq[c], o);
    cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, o);
  }
  if (lane == 0) {
#pragma unroll
    for (int c = 0; c < GHP; ++c) warp_sq[warp][c] = sq[c];
    warp_n[warp] = cnt;
  }
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
  for (int j = lo + tid; j < hi; j += kThreads) {
    const bool keep_always = p.mask != nullptr && p.mask[j] != 0;
    float sum = 0.0f;
#pragma unroll
    for (int c = 0; c < GHP; ++c) {
      if (c < H) {
        const size_t e = static_cast<size_t>(j) * H + c;
        const float v = keep_always ? 0.0f : p.s[e] * inv[c];
        p.b_out[e] = v;
        sum += v;
      }
    }
    if (GHP > 1 && p.b_sel != nullptr) p.b_sel[j] = sum / static_cast<float>(H);
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
