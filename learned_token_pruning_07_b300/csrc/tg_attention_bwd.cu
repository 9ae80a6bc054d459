// tg_attention_bwd.cu — backward of token-gated attention (TokenGate deep dive, section 3.2:
// the gate score reaches the loss only through the per-key attention bias, Eq. (5)/(8); the
// top-K choice itself carries no gradient, section 3.1), and the gate-score gradient.
//
// For one sequence and query head h (kv head h / group), with x_ij = tau_h q_i.k_j / sqrt(d_h)
// + beta_h ln g_j over j <= i and P_ij = exp(x_ij - LSE_i) (LSE from the forward):
//   dP_ij = dO_i . v_j,  D_i = dO_i . o_i,  dX_ij = P_ij (dP_ij - D_i)
//   dV_j = sum_i P_ij dO_i,  dK_j = tau_h / sqrt(d_h) sum_i dX_ij q_i,
//   dQ_i = tau_h / sqrt(d_h) sum_j dX_ij k_j,  dbias_jh = sum_i dX_ij.
//
// This first version runs on the CUDA cores in fp32: 64x64 tiles of S, P, dP and dX are
// recomputed in shared memory by two kernels, one per key tile (dK, dV, dbias; the query heads
// of a GQA group add into their kv head's dK, dV in head order) and one per query tile (dQ).
// Every output element is written by exactly one CTA after a fixed-order sum: deterministic,
// no atomics and no scratch memory.
#include "tg_common.cuh"

namespace {

constexpr int kT = 64;         // rows per tile (queries or keys)
constexpr int kThreads = 256;  // 16 x 16 threads; a thread owns a 4 x 4 block of a 64 x 64 tile
constexpr int kMaxHeads = 128;

struct BwdParams {
  const uint16_t *Q, *K, *V, *O, *dO;
  const float *g;
  int32_t g_cols, g_group;  // gate heads per row (H_g); query heads per gate head
  const float *lse;
  const int32_t *cu_kept;
  int32_t B, M_cap, H_q, H_kv, group, n_tiles;
  float *dQ, *dK, *dV, *dbias;
  int32_t *status;
  float scale[kMaxHeads];  // tau_h / sqrt(d_h)
  float beta[kMaxHeads];
};

template <int D>
struct BwdSmem {
  static constexpr int kPitch = D + 1;  // padded rows: conflict-light column walks
  float q[kT][kPitch];   // query-side rows: Q (dkdv) or Q (dq)
  float dO[kT][kPitch];
  float k[kT][kPitch];
  float v[kT][kPitch];
  float p[kT][kT + 1];   // P
  float x[kT][kT + 1];   // dX
  float lse[kT], dd[kT], bias[kT];
};

__device__ __forceinline__ float bf(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// Load `kT` rows of head `head` of a [M, H, D] bf16 tensor into fp32 shared rows (zeros past n).
template <int D>
__device__ __forceinline__ void load_rows(float (*dst)[D + 1], const uint16_t *src, int row0, int n,
                                          int H, int head) {
  for (int e = threadIdx.x; e < kT * D; e += kThreads) {
    const int r = e / D, c = e % D;
    dst[r][c] = r < n ? bf(src[(static_cast<size_t>(row0 + r) * H + head) * D + c]) : 0.0f;
  }
}

// Sequence boundaries for tile `tile` of sequence b; false if the tile is past the end.
__device__ __forceinline__ bool tile_bounds(const BwdParams &p, int b, int tile, int &start, int &len) {
  int s0 = p.cu_kept[b], s1 = p.cu_kept[b + 1];
  if (s0 < 0 || s1 < s0) {
    if (threadIdx.x == 0 && tile == 0) tg::report(p.status, TG_DEV_BAD_SEQLENS);
    return false;
  }
  s0 = min(s0, p.M_cap);
  s1 = min(s1, p.M_cap);
  start = s0;
  len = s1 - s0;
  return tile * kT < len;
}

// S, P, dP and dX of query tile [qi0, qi0 + nq) against key tile [kj0, kj0 + nk) of one
// sequence (positions relative to its start), for query head h. sm.q/dO/k/v, lse, dd (D_i) and
// bias hold the tiles. Leaves P in sm.p and dX in sm.x.
template <int D>
__device__ __forceinline__ void tile_grads(BwdSmem<D> &sm, int qi0, int nq, int kj0, int nk, float scale) {
  const int ti = threadIdx.x / 16, tj = threadIdx.x % 16;
  float s[4][4] = {}, dp[4][4] = {};
  for (int c = 0; c < D; ++c) {
    float a[4], bq[4], bk[4], bv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      a[i] = sm.q[4 * ti + i][c];
      bq[i] = sm.dO[4 * ti + i][c];
      bk[i] = sm.k[4 * tj + i][c];
      bv[i] = sm.v[4 * tj + i][c];
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        s[i][j] = fmaf(a[i], bk[j], s[i][j]);
        dp[i][j] = fmaf(bq[i], bv[j], dp[i][j]);
      }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 4 * ti + i;
    const float lse = sm.lse[r];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = 4 * tj + j;
      // visible: both inside the sequence and key position <= query position
      const bool vis = r < nq && c < nk && kj0 + c <= qi0 + r && lse != -INFINITY;
      const float pr = vis ? expf(fmaf(scale, s[i][j], sm.bias[c]) - lse) : 0.0f;
      sm.p[r][c] = pr;
      sm.x[r][c] = pr * (dp[i][j] - sm.dd[r]);
    }
  }
}

// D_i = dO_i . o_i and LSE_i of query tile rows, for head h.
template <int D>
__device__ __forceinline__ void row_terms(BwdSmem<D> &sm, const BwdParams &p, int row0, int nq, int h) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int r = warp; r < kT; r += kThreads / 32) {
    float acc = 0.0f;
    if (r < nq) {
      const uint16_t *orow = p.O + (static_cast<size_t>(row0 + r) * p.H_q + h) * D;
      for (int c = lane; c < D; c += 32) acc = fmaf(sm.dO[r][c], bf(orow[c]), acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    if (lane == 0) {
      sm.dd[r] = acc;
      sm.lse[r] = r < nq ? p.lse[static_cast<size_t>(row0 + r) * p.H_q + h] : -INFINITY;
    }
  }
}

// Per-key bias beta_h ln g_j of a key tile (0 where beta_h = 0, as in the forward).
template <int D>
__device__ __forceinline__ void key_bias(BwdSmem<D> &sm, const BwdParams &p, int row0, int nk, int h) {
  for (int c = threadIdx.x; c < kT; c += kThreads) {
    float b = 0.0f;
    if (p.g != nullptr && p.beta[h] != 0.0f && c < nk)
      b = p.beta[h] * logf(p.g[static_cast<size_t>(row0 + c) * p.g_cols + h / p.g_group]);
    sm.bias[c] = b;
  }
}

// ---- key tiles: dK, dV (kv head) and dbias (every query head of the group) ----
template <int D>
__global__ void __launch_bounds__(kThreads, 1) bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  BwdSmem<D> &sm = *reinterpret_cast<BwdSmem<D> *>(smem_raw);
  tg::pdl_wait();
  tg::pdl_launch_dependents();
  const int kvh = blockIdx.x % p.H_kv;
  const int rest = blockIdx.x / p.H_kv;
  const int b = rest % p.B;
  const int kt = rest / p.B;
  int start, len;
  if (!tile_bounds(p, b, kt, start, len)) return;
  const int kj0 = kt * kT, nk = min(kT, len - kj0);
  load_rows<D>(sm.k, p.K, start + kj0, nk, p.H_kv, kvh);
  load_rows<D>(sm.v, p.V, start + kj0, nk, p.H_kv, kvh);
  // output block of this thread: keys 4*tc .. +3, features kF*td .. +kF-1 (16 x kF = D)
  constexpr int kF = D / 16;
  const int tc = threadIdx.x / 16, td = threadIdx.x % 16;
  float dk[4][kF] = {}, dv[4][kF] = {};
  const int n_qt = (len + kT - 1) / kT;
  for (int gi = 0; gi < p.group; ++gi) {
    const int h = kvh * p.group + gi;
    const float scale = p.scale[h];
    float dbias = 0.0f;  // threads 0..63: the column sum of dX for key threadIdx.x
    __syncthreads();
    key_bias<D>(sm, p, start + kj0, nk, h);
    for (int qt = kt; qt < n_qt; ++qt) {  // causal: query tiles at or after the key tile
      const int qi0 = qt * kT, nq = min(kT, len - qi0);
      __syncthreads();
      load_rows<D>(sm.q, p.Q, start + qi0, nq, p.H_q, h);
      load_rows<D>(sm.dO, p.dO, start + qi0, nq, p.H_q, h);
      __syncthreads();
      row_terms<D>(sm, p, start + qi0, nq, h);
      __syncthreads();
      tile_grads<D>(sm, qi0, nq, kj0, nk, scale);
      __syncthreads();
      for (int r = 0; r < kT; ++r) {
        float pr[4], xr[4], dor[kF], qr[kF];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          pr[i] = sm.p[r][4 * tc + i];
          xr[i] = sm.x[r][4 * tc + i];
        }
#pragma unroll
        for (int f = 0; f < kF; ++f) {
          dor[f] = sm.dO[r][kF * td + f];
          qr[f] = sm.q[r][kF * td + f];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int f = 0; f < kF; ++f) {
            dv[i][f] = fmaf(pr[i], dor[f], dv[i][f]);
            dk[i][f] = fmaf(xr[i] * scale, qr[f], dk[i][f]);
          }
      }
      if (threadIdx.x < kT)
        for (int r = 0; r < kT; ++r) dbias += sm.x[r][threadIdx.x];
    }
    if (threadIdx.x < nk) p.dbias[static_cast<size_t>(start + kj0 + threadIdx.x) * p.H_q + h] = dbias;
  }
  for (int i = 0; i < 4; ++i) {
    const int c = 4 * tc + i;
    if (c >= nk) continue;
    const size_t base = (static_cast<size_t>(start + kj0 + c) * p.H_kv + kvh) * D + kF * td;
    for (int f = 0; f < kF; ++f) {
      p.dK[base + f] = dk[i][f];
      p.dV[base + f] = dv[i][f];
    }
  }
}

// ---- query tiles: dQ ----
template <int D>
__global__ void __launch_bounds__(kThreads, 1) bwd_dq_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  BwdSmem<D> &sm = *reinterpret_cast<BwdSmem<D> *>(smem_raw);
  tg::pdl_wait();
  tg::pdl_launch_dependents();
  const int h = blockIdx.x % p.H_q;
  const int rest = blockIdx.x / p.H_q;
  const int b = rest % p.B;
  const int qt = rest / p.B;
  int start, len;
  if (!tile_bounds(p, b, qt, start, len)) return;
  const int kvh = h / p.group;
  const float scale = p.scale[h];
  const int qi0 = qt * kT, nq = min(kT, len - qi0);
  load_rows<D>(sm.q, p.Q, start + qi0, nq, p.H_q, h);
  load_rows<D>(sm.dO, p.dO, start + qi0, nq, p.H_q, h);
  __syncthreads();
  row_terms<D>(sm, p, start + qi0, nq, h);
  constexpr int kF = D / 16;  // features per thread: 16 x kF = D
  const int tr = threadIdx.x / 16, td = threadIdx.x % 16;
  float dq[4][kF] = {};
  for (int kt = 0; kt <= qt; ++kt) {  // causal: key tiles at or before the query tile
    const int kj0 = kt * kT, nk = min(kT, len - kj0);
    __syncthreads();
    load_rows<D>(sm.k, p.K, start + kj0, nk, p.H_kv, kvh);
    load_rows<D>(sm.v, p.V, start + kj0, nk, p.H_kv, kvh);
    key_bias<D>(sm, p, start + kj0, nk, h);
    __syncthreads();
    tile_grads<D>(sm, qi0, nq, kj0, nk, scale);
    __syncthreads();
    for (int c = 0; c < kT; ++c) {
      float xr[4], kr[kF];
#pragma unroll
      for (int i = 0; i < 4; ++i) xr[i] = sm.x[4 * tr + i][c];
#pragma unroll
      for (int f = 0; f < kF; ++f) kr[f] = sm.k[c][kF * td + f];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int f = 0; f < kF; ++f) dq[i][f] = fmaf(xr[i], kr[f], dq[i][f]);
    }
  }
  for (int i = 0; i < 4; ++i) {
    const int r = 4 * tr + i;
    if (r >= nq) continue;
    const size_t base = (static_cast<size_t>(start + qi0 + r) * p.H_q + h) * D + kF * td;
    for (int f = 0; f < kF; ++f) p.dQ[base + f] = dq[i][f] * scale;
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

template <int D>
tg_status launch_bwd_d(const BwdParams &p, int n_tiles, cudaStream_t stream) {
  const int smem = static_cast<int>(sizeof(BwdSmem<D>));
  cudaError_t e = cudaFuncSetAttribute(bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return tg_host::record_cuda(e);
  const long long g_kv = static_cast<long long>(n_tiles) * p.B * p.H_kv;
  const long long g_q = static_cast<long long>(n_tiles) * p.B * p.H_q;
  if (g_q > 0x7FFFFFFFLL) return TG_ERR_UNSUPPORTED;
  e = tg_host::launch_pdl(bwd_dkdv_kernel<D>, dim3(static_cast<int>(g_kv)), dim3(kThreads), smem, stream, p);
  if (e == cudaSuccess)
    e = tg_host::launch_pdl(bwd_dq_kernel<D>, dim3(static_cast<int>(g_q)), dim3(kThreads), smem, stream, p);
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
  p.Q = Q;
  p.K = K;
  p.V = V;
  p.O = O;
  p.dO = dO;
  p.g = g;
  p.g_cols = H_g;
  p.g_group = H_q / H_g;
  p.lse = lse;
  p.cu_kept = cu_kept;
  p.B = B;
  p.M_cap = M_cap;
  p.H_q = H_q;
  p.H_kv = H_kv;
  p.group = H_q / H_kv;
  p.dQ = dQ;
  p.dK = dK;
  p.dV = dV;
  p.dbias = dbias;
  p.status = status;
  const int n_tiles = (max_seqlen + kT - 1) / kT;
  p.n_tiles = n_tiles;
  for (int h = 0; h < kMaxHeads; ++h) {
    p.scale[h] = h < H_q ? tau[h] / std::sqrt(static_cast<float>(d_h)) : 0.0f;
    p.beta[h] = h < H_q ? beta[h] : 0.0f;
  }
  if (d_h == 128) return launch_bwd_d<128>(p, n_tiles, stream);
  if (d_h == 64) return launch_bwd_d<64>(p, n_tiles, stream);
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
