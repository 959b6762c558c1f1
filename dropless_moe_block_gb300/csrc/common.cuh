// Shared host/device helpers of the dmoe CUDA library (sm_103a only).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <utility>

#include "dmoe.h"

#define DMOE_API extern "C" __attribute__((visibility("default")))

namespace dmoe {

// ----------------------------------------------------------------- host side

struct DeviceInfo {
  int device;
  int sm_count;
  int cc_major, cc_minor;
  int32_t* err_word;  // device address of the library's error word
};

// Current device's properties; returns DMOE_ERR_CUDA / DMOE_ERR_UNSUPPORTED
// when the device cannot be queried or is not compute capability 10.3.
dmoe_status device_info(DeviceInfo* out);

// Adds n to the process-wide launch counter.
void count_launches(int n);

// Maps the last CUDA error to a status (clears it).
dmoe_status cuda_status(cudaError_t e);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline cudaStream_t as_stream(dmoe_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// Launches kern<<<grid, block, smem, st>>>(args...) with programmatic stream
// serialization, so that it may overlap the tail of the previous kernel.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// As launch_pdl, in thread-block clusters of cluster_x CTAs along x (grid.x a
// multiple of cluster_x).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                               int cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(cluster_x);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ------------------------------------------------------------- device side

// Global-timer based limit for every spin-wait (1 s).
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may start while the previous kernel on the
// stream is still running; pdl_wait() blocks until that kernel has completed
// and its memory is visible (a no-op without a prerequisite grid), and
// pdl_launch_dependents() lets the next such kernel start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Records the first error of the process (sticky until cleared by the host).
__device__ __forceinline__ void raise_error(int32_t* err, int32_t code) {
  if (err) atomicCAS(err, 0, code);
}

}  // namespace dmoe
