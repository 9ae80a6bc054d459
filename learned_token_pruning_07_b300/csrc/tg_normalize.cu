// tg_normalize.cu — sequence-axis RMS normalisation of the gate scores (TokenGate deep dive,
// section 3.1, Eq. (3)): b_j = s_j / sqrt(mean over the sequence's prunable rows of s^2 + eps),
// and b_j = 0 on the non-prunable rows.
//
// One 8-CTA cluster per sequence. Each CTA sums s^2 and counts the prunable rows of its
// contiguous chunk in a fixed order (per thread in index order, then a shuffle tree per warp,
// then the warps in order); the cluster adds the eight partial sums in rank order through
// distributed shared memory, so the result does not depend on timing. Then every CTA writes
// the normalised scores of its chunk.
#include <cooperative_groups.h>

#include "tg_common.cuh"

namespace cg = cooperative_groups;

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kCluster = 8;

struct NormParams {
  const float *s;
  const uint8_t *mask;
  const int32_t *cu_seqlens;
  int32_t B, T;
  float eps;
  float *b_out;
  int32_t *status;
};

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, 1)
    normalize_scores_kernel(const __grid_constant__ NormParams p) {
  __shared__ float warp_sq[kWarps];
  __shared__ int32_t warp_n[kWarps];
  __shared__ float cta_sq;
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

  float sq = 0.0f;
  int cnt = 0;
  for (int j = lo + tid; j < hi; j += kThreads) {
    if (p.mask == nullptr || p.mask[j] == 0) {
      const float v = p.s[j];
      sq = fmaf(v, v, sq);
      ++cnt;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sq += __shfl_xor_sync(0xFFFFFFFFu, sq, o);
    cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, o);
  }
  if (lane == 0) {
    warp_sq[warp] = sq;
    warp_n[warp] = cnt;
  }
  __syncthreads();
  if (tid == 0) {
    float t = 0.0f;
    int c = 0;
    for (int w = 0; w < kWarps; ++w) {
      t += warp_sq[w];
      c += warp_n[w];
    }
    cta_sq = t;
    cta_n = c;
  }
  cluster.sync();
  float total = 0.0f;
  int n_doc = 0;
  for (int r = 0; r < kCluster; ++r) {  // rank order: the same sum in every CTA
    total += *cluster.map_shared_rank(&cta_sq, r);
    n_doc += *cluster.map_shared_rank(&cta_n, r);
  }
  // a sequence without prunable rows has nothing to scale: every b is 0
  const float inv = n_doc > 0 ? 1.0f / sqrtf(total / static_cast<float>(n_doc) + p.eps) : 0.0f;
  for (int j = lo + tid; j < hi; j += kThreads) {
    const bool keep_always = p.mask != nullptr && p.mask[j] != 0;
    p.b_out[j] = keep_always ? 0.0f : p.s[j] * inv;
  }
  cluster.sync();  // keep this CTA's shared memory alive until every peer has read it
}

}  // namespace

namespace tg_host {

tg_status launch_normalize_scores(const float *s, const uint8_t *mask, const int32_t *cu_seqlens,
                                  int32_t B, int32_t T, float eps, float *b_out, int32_t *status,
                                  cudaStream_t stream) {
  NormParams p{s, mask, cu_seqlens, B, T, eps, b_out, status};
  return record_cuda(launch_pdl(normalize_scores_kernel, dim3(B * kCluster), dim3(kThreads), 0, stream, p));
}

}  // namespace tg_host
