// tg_gather.cu — slice the kept rows (TokenGate deep dive, section 3.4: hidden_states[:, keep]
// and position_ids[:, keep], the original position ids) and carry each kept token's gate
// value (or its H_g per-head gate values, section 3.4) with it (TokenGate paper page,
// Figure 1 (b)); plus RoPE at the gathered original positions.
//
// Gather: one warp per kept row, 16-byte vector loads and streaming stores; the grid is a
// fixed multiple of the SM count and strides over rows, so it needs no host knowledge of
// the kept count M (read from cu_kept[B] on the device).
#include "tg_common.cuh"

namespace {

constexpr int kGatherThreads = 256;
constexpr int kGatherWarps = kGatherThreads / 32;

struct GatherParams {
  const uint16_t *h;
  const int32_t *pos;
  const float *g;
  int32_t H_g;  // gate values per row (per-head gates: H_g <= 32, one lane each)
  const int32_t *cu_seqlens;
  int32_t B, T, d;
  int32_t B_kept;  // cu_kept has B_kept + 1 entries (B for one list; 2B for a two-budget pack)
  const int32_t *kept_idx;
  const int32_t *cu_kept;
  int32_t capacity;
  uint16_t *h_kept;
  int32_t *pos_kept;
  float *g_kept;
  int32_t *status;
};

__global__ void __launch_bounds__(kGatherThreads) gather_kernel(GatherParams p) {
  tg::pdl_wait();
  tg::pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int nvec = p.d >> 3;  // 16-byte vectors per row
  const int stride = gridDim.x * kGatherWarps;
  const int m0 = blockIdx.x * kGatherWarps + (threadIdx.x >> 5);
  // the first row's index is fetched together with the kept count (both sit in L2 from the
  // selection); an index at m >= M is read from inside the buffer but never used
  int j_next = m0 < p.capacity ? p.kept_idx[m0] : -1;
  int M = min(p.cu_kept[p.B_kept], p.capacity);
  if (M < 0) M = 0;
  for (int m = m0; m < M; m += stride) {
    const int j = j_next;
    if (m + stride < M) j_next = p.kept_idx[m + stride];
    if (j < 0 || j >= p.T) {
      if (lane == 0) tg::report(p.status, TG_DEV_BAD_INDEX);
      continue;
    }
    tg::warp_copy_row(reinterpret_cast<uint4 *>(p.h_kept + static_cast<size_t>(m) * p.d),
                      reinterpret_cast<const uint4 *>(p.h + static_cast<size_t>(j) * p.d), nvec, lane);
    if (lane == 0) {
      if (p.pos_kept) {
        int pv;
        if (p.pos) {
          pv = p.pos[j];
        } else {
          int lo_b = 0, hi_b = p.B;  // largest b with cu_seqlens[b] <= j
          while (hi_b - lo_b > 1) {
            const int mid = (lo_b + hi_b) >> 1;
            if (p.cu_seqlens[mid] <= j) lo_b = mid; else hi_b = mid;
          }
          pv = j - p.cu_seqlens[lo_b];
        }
        p.pos_kept[m] = pv;
      }
    }
    if (p.g_kept && p.g && lane < p.H_g)
      p.g_kept[static_cast<size_t>(m) * p.H_g + lane] = p.g[static_cast<size_t>(j) * p.H_g + lane];
  }
}

// ---------------------------------------------------------------------------
// Two-budget packing: the full budget keeps every row, so its half of the packed keep list is
// the identity and its boundaries are the input's.
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(256) two_budget_prologue_kernel(const int32_t *cu_seqlens, int32_t B,
                                                                   int32_t T, int32_t *kept_idx,
                                                                   int32_t *cu_packed) {
  tg::pdl_wait();
  tg::pdl_launch_dependents();
  const int stride = gridDim.x * 256;
  for (int i = blockIdx.x * 256 + threadIdx.x; i < T; i += stride) kept_idx[i] = i;
  for (int i = blockIdx.x * 256 + threadIdx.x; i <= B; i += stride) cu_packed[i] = cu_seqlens[i];
}

// ---------------------------------------------------------------------------
// RoPE (rotate-half): pairs (x_i, x_{i+d_h/2}) of every head of a row rotate by
// pos * inv_freq_i. The angle is formed and reduced modulo 2*pi in fp64 (positions reach
// 10^5, where an fp32 angle would be off by ~1e-2 rad), then sin/cos run in fp32.
// ---------------------------------------------------------------------------

constexpr int kMaxHalf = 128;

struct RopeParams {
  uint16_t *X;
  const int32_t *pos;
  const int32_t *cu_kept;
  int32_t B, capacity, H, d_h;
  double inv_freq[kMaxHalf];
};

__global__ void __launch_bounds__(256) rope_kernel(const __grid_constant__ RopeParams p) {
  tg::pdl_wait();
  tg::pdl_launch_dependents();
  int M = p.capacity;
  if (p.cu_kept) M = max(0, min(p.cu_kept[p.B], p.capacity));
  const int half = p.d_h >> 1;
  const long long total = static_cast<long long>(M) * half;
  const double two_pi = 6.283185307179586476925286766559;
  for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < total;
       t += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int m = static_cast<int>(t / half);
    const int i = static_cast<int>(t % half);
    const double ang = static_cast<double>(p.pos[m]) * p.inv_freq[i];
    const double red = ang - two_pi * rint(ang / two_pi);
    float sn, cs;
    sincosf(static_cast<float>(red), &sn, &cs);
    uint16_t *row = p.X + static_cast<size_t>(m) * p.H * p.d_h;
    for (int hh = 0; hh < p.H; ++hh) {
      uint16_t *x = row + hh * p.d_h;
      const float x1 = tg::bf16_bits_to_float(x[i]);
      const float x2 = tg::bf16_bits_to_float(x[i + half]);
      x[i] = tg::float_to_bf16_bits(x1 * cs - x2 * sn);
      x[i + half] = tg::float_to_bf16_bits(x2 * cs + x1 * sn);
    }
  }
}

}  // namespace

namespace tg_host {

tg_status launch_gather(const uint16_t *h, const int32_t *pos, const float *g, int32_t H_g,
                        const int32_t *cu_seqlens, int32_t B, int32_t T, int32_t d,
                        const int32_t *kept_idx, const int32_t *cu_kept, int32_t capacity,
                        uint16_t *h_kept, int32_t *pos_kept, float *g_kept, int32_t *status,
                        cudaStream_t stream, int32_t B_kept) {
  if (capacity == 0) return TG_OK;
  GatherParams p{h, pos, g, H_g, cu_seqlens, B, T, d, B_kept < 0 ? B : B_kept, kept_idx, cu_kept, capacity,
                 h_kept, pos_kept, g_kept, status};
  int grid = (capacity + kGatherWarps - 1) / kGatherWarps;
  if (grid > num_sms() * 8) grid = num_sms() * 8;
  return record_cuda(launch_pdl(gather_kernel, dim3(grid), dim3(kGatherThreads), 0, stream, p));
}

tg_status launch_two_budget_prologue(const int32_t *cu_seqlens, int32_t B, int32_t T, int32_t *kept_idx,
                                     int32_t *cu_packed, cudaStream_t stream) {
  int grid = (T + 255) / 256;
  if (grid < 1) grid = 1;
  if (grid > num_sms() * 4) grid = num_sms() * 4;
  return record_cuda(launch_pdl(two_budget_prologue_kernel, dim3(grid), dim3(256), 0, stream, cu_seqlens, B, T,
                                kept_idx, cu_packed));
}

tg_status launch_rope(uint16_t *X, const int32_t *pos, const int32_t *cu_kept, int32_t B,
                      int32_t capacity, int32_t H, int32_t d_h, float theta,
                      cudaStream_t stream) {
  if (capacity == 0) return TG_OK;
  RopeParams p;
  p.X = X;
  p.pos = pos;
  p.cu_kept = cu_kept;
  p.B = B;
  p.capacity = capacity;
  p.H = H;
  p.d_h = d_h;
  const int half = d_h / 2;
  for (int i = 0; i < kMaxHalf; ++i)
    p.inv_freq[i] = i < half ? std::pow(static_cast<double>(theta), -2.0 * i / d_h) : 0.0;
  const long long total = static_cast<long long>(capacity) * half;
  long long grid = (total + 255) / 256;
  if (grid > num_sms() * 16) grid = num_sms() * 16;
  return record_cuda(launch_pdl(rope_kernel, dim3(static_cast<int>(grid)), dim3(256), 0, stream, p));
}

}  // namespace tg_host
