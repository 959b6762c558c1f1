// Utility entry points of the C ABI: version, status strings, the device
// error word and the launch counter.
#include <atomic>
#include <mutex>

#include "common.cuh"

namespace {

__device__ int32_t g_err_word;  // sticky device error word, one per device
__device__ int32_t g_never_set;  // a flag that no kernel of the library sets

// One warp waits on g_never_set with the bounded spin of the library's
// kernels (%globaltimer limit, checked every 32 tries), then reports the
// timeout through the error word and returns.
__global__ void selftest_wait_kernel(uint64_t limit_ns, int32_t* err) {
  const uint64_t t0 = dmoe::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (*reinterpret_cast<volatile int32_t*>(&g_never_set) != 0) return;
    if ((it & 31u) == 0 && dmoe::globaltimer_ns() - t0 > limit_ns) break;
    __nanosleep(128);
  }
  if (threadIdx.x == 0) dmoe::raise_error(err, DMOE_SITE_SELFTEST | DMOE_ERR_TIMEOUT);
}

std::atomic<int64_t> g_launches{0};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
bool g_have[kMaxDevices];
dmoe::DeviceInfo g_info[kMaxDevices];

}  // namespace

namespace dmoe {

void count_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

dmoe_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return DMOE_OK;
  (void)cudaGetLastError();
  return DMOE_ERR_CUDA;
}

dmoe_status device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cuda_status(cudaErrorUnknown);
  if (dev < 0 || dev >= kMaxDevices) return DMOE_ERR_UNSUPPORTED;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_have[dev]) {
      *out = g_info[dev];
      return DMOE_OK;
    }
  }
  DeviceInfo d{};
  d.device = dev;
  if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return cuda_status(cudaErrorUnknown);
  if (d.cc_major != 10 || d.cc_minor != 3) return DMOE_ERR_UNSUPPORTED;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return cuda_status(cudaErrorUnknown);
  d.err_word = static_cast<int32_t*>(p);
  std::lock_guard<std::mutex> lk(g_mu);
  g_info[dev] = d;
  g_have[dev] = true;
  *out = d;
  return DMOE_OK;
}

}  // namespace dmoe

DMOE_API const char* dmoe_version(void) { return "dmoe 0.1.0 (sm_103a, tcgen05/TMA)"; }

DMOE_API const char* dmoe_status_string(int status) {
  switch (status & 0xff) {
    case DMOE_OK: return "ok";
    case DMOE_ERR_INVALID_ARG: return "invalid argument";
    case DMOE_ERR_UNSUPPORTED: return "unsupported (needs an sm_103 GPU)";
    case DMOE_ERR_CUDA: return "CUDA error";
    case DMOE_ERR_TIMEOUT: return "a bounded device wait gave up";
    case DMOE_ERR_DEVICE: return "invalid data found on the device";
    default: return "unknown status";
  }
}

DMOE_API int64_t dmoe_padded_rows_max_block(int T, int k, int E, int block) {
  if (T < 0 || k < 1 || E < 1 || (block != 64 && block != 128 && block != 256)) return -1;
  const int64_t A = int64_t(T) * k;
  const int64_t live = A < E ? A : E;
  return ((A + live * (block - 1)) / block) * block;
}

DMOE_API int64_t dmoe_padded_rows_max(int T, int k, int E) { return dmoe_padded_rows_max_block(T, k, E, DMOE_BLOCK); }

DMOE_API int64_t dmoe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

DMOE_API dmoe_status dmoe_get_error(int32_t* code_out, int clear) {
  if (!code_out) return DMOE_ERR_INVALID_ARG;
  dmoe::DeviceInfo di;
  dmoe_status s = dmoe::device_info(&di);
  if (s != DMOE_OK) return s;
  if (cudaDeviceSynchronize() != cudaSuccess) return dmoe::cuda_status(cudaErrorUnknown);
  int32_t v = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_word, sizeof(v)) != cudaSuccess) return dmoe::cuda_status(cudaErrorUnknown);
  *code_out = v;
  if (clear) {
    const int32_t z = 0;
    if (cudaMemcpyToSymbol(g_err_word, &z, sizeof(z)) != cudaSuccess) return dmoe::cuda_status(cudaErrorUnknown);
  }
  return DMOE_OK;
}

DMOE_API dmoe_status dmoe_selftest_bounded_wait(int64_t limit_ns, dmoe_stream_t stream) {
  if (limit_ns < 1000 || limit_ns > static_cast<int64_t>(dmoe::kWaitLimitNs)) return DMOE_ERR_INVALID_ARG;
  dmoe::DeviceInfo di;
  dmoe_status s = dmoe::device_info(&di);
  if (s != DMOE_OK) return s;
  selftest_wait_kernel<<<1, 32, 0, dmoe::as_stream(stream)>>>(static_cast<uint64_t>(limit_ns), di.err_word);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return dmoe::cuda_status(e);
  dmoe::count_launches(1);
  return DMOE_OK;
}
