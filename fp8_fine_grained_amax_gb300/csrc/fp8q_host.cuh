// fp8q_host.cuh -- host-side helpers shared by the entry points: device
// checks, argument validation and launch error mapping.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "fp8q.h"

namespace fp8q {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool checked = false;
  bool supported = false;
  int sm_count = 0;
  int max_smem_optin = 0;
};

// Per-device properties, read once.  The library only runs on sm_103 parts.
inline fp8q_status device_info(DeviceInfo &out) {
  static DeviceInfo table[kMaxDevices];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FP8Q_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FP8Q_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(mu);
  DeviceInfo &d = table[dev];
  if (!d.checked) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess)
      return FP8Q_ERR_CUDA;
    d.supported = (major == 10 && minor == 3);
    d.checked = true;
  }
  out = d;
  return d.supported ? FP8Q_OK : FP8Q_ERR_UNSUPPORTED;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

inline fp8q_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA;
}

}  // namespace fp8q
