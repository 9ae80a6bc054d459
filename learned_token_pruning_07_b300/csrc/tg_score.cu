// tg_score.cu — gate scoring (TokenGate deep dive, section 3.1, Eq. (3): b~_j = MLP(a~_j)).
//
// One CTA owns a 128-row tile of hidden states and the full d_g-wide hidden layer of the
// score MLP. The d-reduction u = h W1^T runs on the tensor cores (tcgen05.mma kind::f16,
// bf16 operands staged by TMA into 64-byte-swizzled shared memory, fp32 accumulator in
// tensor memory: 128 lanes x d_g columns). The epilogue reads each row's accumulator
// out of tensor memory and finishes the MLP in fp32 registers:
//   s = w2 . SiLU(u + b1) + b2,  g = sigmoid(s)  (g = 1 on non-prunable rows).
// Roles: warp 0 lane 0 issues TMA, warp 1 lane 0 issues MMAs, warp 2 owns the tensor-memory
// allocation, all four warps run the epilogue (warp w reads TMEM lanes 32w..32w+31).
#include "tg_common.cuh"

namespace {

constexpr int kBM = 128;      // rows per tile = tensor-memory lanes
constexpr int kBK = 32;       // d-elements per pipeline stage (one 64-byte swizzled row)
constexpr int kStages = 5;
constexpr int kThreads = 128;
constexpr int kMaxDg = 512;

struct ScoreParams {
  int32_t T, d, d_g, n_inst, n_split;
  uint32_t tmem_cols;
  const float *b1;
  const uint16_t *w2;
  float b2;
  const uint8_t *mask;
  float *s_out;
  float *g_out;
  int32_t *status;
  uint64_t wait_limit;
};

struct SmemLayout {
  uint32_t a_bytes, b_bytes, off_b, off_w2, off_b1, off_bar, total;
};

__host__ __device__ inline SmemLayout score_smem_layout(int d_g) {
  SmemLayout L;
  L.a_bytes = kBM * kBK * 2;
  L.b_bytes = static_cast<uint32_t>(d_g) * kBK * 2;
  L.off_b = kStages * L.a_bytes;
  L.off_w2 = L.off_b + kStages * L.b_bytes;
  L.off_b1 = L.off_w2 + kMaxDg * 4;
  L.off_bar = L.off_b1 + kMaxDg * 4;
  L.total = L.off_bar + 256 + 1024;  // barriers + slots, plus alignment slack
  return L;
}

__global__ void __launch_bounds__(kThreads, 1)
    gate_score_kernel(const __grid_constant__ CUtensorMap tm_h,
                      const __grid_constant__ CUtensorMap tm_w, ScoreParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const SmemLayout L = score_smem_layout(p.d_g);
  uint8_t *sA = smem;
  uint8_t *sB = smem + L.off_b;
  float *s_w2 = reinterpret_cast<float *>(smem + L.off_w2);
  float *s_b1 = reinterpret_cast<float *>(smem + L.off_b1);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.off_bar);
  uint64_t *empty = full + kStages;
  uint64_t *accum = empty + kStages;
  uint64_t *drain = accum + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  int32_t *abort_flag = reinterpret_cast<int32_t *>(tmem_slot + 1);
  int32_t *n_issued = abort_flag + 1;
  int32_t *n_consumed = abort_flag + 2;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      tg::mbar_init(&full[i], 1);
      tg::mbar_init(&empty[i], 1);
    }
    tg::mbar_init(accum, 1);
    tg::mbar_init(drain, 1);
    *abort_flag = 0;
    *n_issued = 0;
    *n_consumed = 0;
    tg::fence_mbar_init();
    tg::prefetch_tensormap(&tm_h);
    tg::prefetch_tensormap(&tm_w);
  }
  if (warp == 2) {
    tg::tmem_alloc(tmem_slot, p.tmem_cols);
    tg::tmem_relinquish();
  }
  for (int i = threadIdx.x; i < p.d_g; i += kThreads) {
    s_w2[i] = tg::bf16_bits_to_float(p.w2[i]);
    s_b1[i] = p.b1 ? p.b1[i] : 0.0f;
  }
  tg::tc_fence_before();
  __syncthreads();
  tg::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int row0 = blockIdx.x * kBM;
  const int KT = p.d / kBK;
  volatile int32_t *vabort = abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      // TMA producer: fill stage st with the h tile [128 x 32] and W1 slice [d_g x 32].
      int issued = 0;
      for (int kt = 0; kt < KT; ++kt) {
        const int st = kt % kStages;
        const uint32_t ph = (kt / kStages) & 1;
        if (!tg::mbar_wait(&empty[st], ph ^ 1u, vabort, p.wait_limit)) {
          *vabort = 1;
          break;
        }
        tg::mbar_arrive_expect_tx(&full[st], L.a_bytes + L.b_bytes);
        tg::tma_load_2d(sA + st * L.a_bytes, &tm_h, &full[st], kt * kBK, row0);
        for (int j = 0; j < p.n_split; ++j)
          tg::tma_load_2d(sB + st * L.b_bytes + j * p.n_inst * (kBK * 2), &tm_w, &full[st],
                          kt * kBK, j * p.n_inst);
        issued = kt + 1;
      }
      *n_issued = issued;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // MMA issuer: u[128 x d_g] += A[128 x 16] * B[d_g x 16]^T, two K-steps per stage.
      const uint32_t idesc = tg::idesc_bf16_f32(kBM, p.n_inst);
      int consumed = 0;
      bool ok = true;
      for (int kt = 0; kt < KT; ++kt) {
        const int st = kt % kStages;
        const uint32_t ph = (kt / kStages) & 1;
        if (!tg::mbar_wait(&full[st], ph, vabort, p.wait_limit)) {
          *vabort = 1;
          ok = false;
          break;
        }
        tg::tc_fence_after();
        const uint32_t a_base = tg::smem_u32(sA + st * L.a_bytes);
        const uint32_t b_base = tg::smem_u32(sB + st * L.b_bytes);
#pragma unroll
        for (int ks = 0; ks < kBK / 16; ++ks) {
          const uint64_t a_desc = tg::smem_desc(a_base + ks * 32, 16, 8 * kBK * 2, tg::kSwz64);
          for (int j = 0; j < p.n_split; ++j) {
            const uint64_t b_desc = tg::smem_desc(b_base + j * p.n_inst * (kBK * 2) + ks * 32,
                                                  16, 8 * kBK * 2, tg::kSwz64);
            tg::mma_bf16_ss(tmem + j * p.n_inst, a_desc, b_desc, idesc, (kt | ks) != 0);
          }
        }
        tg::mma_commit(&empty[st]);
        consumed = kt + 1;
      }
      *n_consumed = consumed;
      if (ok) {
        tg::mma_commit(accum);
      } else {
        // drain: wait for the MMAs already issued before the tiles and TMEM go away
        tg::mma_commit(drain);
        volatile int32_t never = 0;
        tg::mbar_wait(drain, 0, &never, p.wait_limit);
      }
    }
  }
  __syncwarp();

  // Epilogue: every thread owns one row of the tile.
  // tcgen05.ld is warp-collective: the whole warp takes the same branch.
  const bool acc_ok = __all_sync(0xffffffffu, tg::mbar_wait(accum, 0, vabort, p.wait_limit));
  tg::tc_fence_after();
  if (acc_ok) {
    const int row = row0 + warp * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    float acc = 0.0f;
    uint32_t r[32];
    for (int c0 = 0; c0 < p.d_g; c0 += 32) {
      tg::tmem_ld_32x32b_x32(lane_base + c0, r);
      tg::tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float u = __uint_as_float(r[i]) + s_b1[c0 + i];
        const float silu = __fdividef(u, 1.0f + __expf(-u));
        acc = fmaf(s_w2[c0 + i], silu, acc);
      }
    }
    if (row < p.T) {
      const float s = acc + p.b2;
      p.s_out[row] = s;
      if (p.g_out) {
        const bool keep_always = p.mask && p.mask[row];
        p.g_out[row] = keep_always ? 1.0f : 1.0f / (1.0f + __expf(-s));
      }
    }
  } else {
    *vabort = 1;
  }

  tg::tc_fence_before();
  __syncthreads();
  if (*vabort) {
    if (threadIdx.x == 0) {
      tg::report(p.status, TG_DEV_TIMEOUT);
      // wait (bounded) for TMA copies that were issued but never consumed
      volatile int32_t never = 0;
      for (int i = *n_consumed; i < *n_issued; ++i)
        tg::mbar_wait(&full[i % kStages], (i / kStages) & 1, &never, p.wait_limit);
    }
    __syncthreads();
  }
  if (warp == 2) {
    tg::tc_fence_after();
    tg::tmem_dealloc(tmem, p.tmem_cols);
  }
}

}  // namespace

namespace tg_host {

tg_status launch_gate_score(const uint16_t *h, int32_t T, int32_t d, const uint8_t *mask,
                            const uint16_t *W1, const float *b1, const uint16_t *w2, float b2,
                            int32_t d_g, float *s_out, float *g_out, int32_t *status,
                            cudaStream_t stream) {
  if (T == 0) return TG_OK;
  ScoreParams p;
  p.T = T;
  p.d = d;
  p.d_g = d_g;
  p.n_split = d_g > 256 ? 2 : 1;
  p.n_inst = d_g / p.n_split;
  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(d_g)) cols <<= 1;
  p.tmem_cols = cols;
  p.b1 = b1;
  p.w2 = w2;
  p.b2 = b2;
  p.mask = mask;
  p.s_out = s_out;
  p.g_out = g_out;
  p.status = status;
  p.wait_limit = wait_limit_ns();

  CUtensorMap tm_h, tm_w;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(d), static_cast<uint64_t>(T)};
    const uint64_t strides[1] = {static_cast<uint64_t>(d) * 2};
    const uint32_t box[2] = {kBK, kBM};
    if (!encode_tmap_bf16(&tm_h, h, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B))
      return TG_ERR_CUDA;
  }
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(d), static_cast<uint64_t>(d_g)};
    const uint64_t strides[1] = {static_cast<uint64_t>(d) * 2};
    const uint32_t box[2] = {kBK, static_cast<uint32_t>(p.n_inst)};
    if (!encode_tmap_bf16(&tm_w, W1, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B))
      return TG_ERR_CUDA;
  }
  const SmemLayout L = score_smem_layout(d_g);
  cudaError_t e = cudaFuncSetAttribute(gate_score_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
  if (e != cudaSuccess) return record_cuda(e);
  const int grid = (T + kBM - 1) / kBM;
  gate_score_kernel<<<grid, kThreads, L.total, stream>>>(tm_h, tm_w, p);
  return record_cuda(cudaGetLastError());
}

}  // namespace tg_host
