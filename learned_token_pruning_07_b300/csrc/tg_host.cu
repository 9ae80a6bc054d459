// tg_host.cu — host-side plumbing shared by the entry points: TMA descriptor encoding
// through the driver entry point (no link-time libcuda dependency, so the library loads
// on machines without a driver), the process-wide wait limit, and status reporting.
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "tg_common.cuh"

namespace {

std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
std::atomic<int32_t> g_withhold{0};
thread_local int32_t g_last_cuda_error = 0;

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
  });
  return fn;
}

}  // namespace

namespace tg_host {

bool encode_tmap_bf16(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                      const uint64_t *strides_bytes, const uint32_t *box,
                      CUtensorMapSwizzle swizzle) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t gdim[5];
  cuuint64_t gstride[4];
  cuuint32_t bdim[5];
  cuuint32_t estride[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estride[i] = 1;
  }
  for (int i = 0; i < rank - 1; ++i) gstride[i] = strides_bytes[i];
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank),
                  const_cast<void *>(base), gdim, gstride, bdim, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

// Waits for a kernel's own copies and MMAs in flight, after a pipeline wait gave up: never
// shorter than 0.2 s, so a small test limit cannot let a CTA exit while a copy still lands.
uint64_t drain_limit_ns() {
  const uint64_t w = wait_limit_ns();
  return w > 200000000ull ? w : 200000000ull;
}

int32_t withhold_mask() { return g_withhold.load(std::memory_order_relaxed); }

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
  return n > 0 ? n : 148;
}

tg_status record_cuda(cudaError_t e) {
  if (e == cudaSuccess) return TG_OK;
  g_last_cuda_error = static_cast<int32_t>(e);
  return TG_ERR_CUDA;
}

}  // namespace tg_host

extern "C" {

int32_t tg_version(void) { return 200; }

const char *tg_status_string(tg_status s) {
  switch (s) {
    case TG_OK: return "ok";
    case TG_ERR_INVALID_ARG: return "invalid argument";
    case TG_ERR_UNSUPPORTED: return "unsupported shape";
    case TG_ERR_CUDA: return "CUDA error";
    case TG_ERR_CAPACITY: return "output capacity exceeded";
    case TG_ERR_DEVICE_TIMEOUT: return "device pipeline wait timed out";
    case TG_ERR_DEVICE: return "device reported invalid input";
    default: return "unknown status";
  }
}

int32_t tg_last_cuda_error(void) { return g_last_cuda_error; }

tg_status tg_set_wait_limit_ns(uint64_t limit_ns) {
  g_wait_limit_ns.store(limit_ns == 0 ? 2000000000ull : limit_ns, std::memory_order_relaxed);
  return TG_OK;
}

tg_status tg_set_test_withhold(int32_t mask) {
  if (mask & ~(TG_WITHHOLD_GATE_SCORE | TG_WITHHOLD_ATTENTION | TG_WITHHOLD_BACKWARD | TG_WITHHOLD_GATE_SCORE_PEER))
    return TG_ERR_INVALID_ARG;
  g_withhold.store(mask, std::memory_order_relaxed);
  return TG_OK;
}

tg_status tg_read_device_status(const int32_t *status, int32_t *out, tg_stream_t stream) {
  if (!status || !out) return TG_ERR_INVALID_ARG;
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, status, sizeof(int32_t), cudaMemcpyDeviceToHost,
                                  reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return tg_host::record_cuda(e);
  *out = v;
  if (v == 0) return TG_OK;
  if (v & TG_DEV_TIMEOUT) return TG_ERR_DEVICE_TIMEOUT;
  if (v == TG_DEV_CAPACITY) return TG_ERR_CAPACITY;
  return TG_ERR_DEVICE;
}

}  // extern "C"
