// Shared host/device helpers of the dmoe CUDA library (sm_103a only).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

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

// ------------------------------------------------------------- device side

// Global-timer based limit for every spin-wait (1 s).
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Records the first error of the process (sticky until cleared by the host).
__device__ __forceinline__ void raise_error(int32_t* err, int32_t code) {
  if (err) atomicCAS(err, 0, code);
}

}  // namespace dmoe
