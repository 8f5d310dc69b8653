// fp8q_host.cuh -- host-side helpers shared by the entry points: device
// checks, argument validation and launch error mapping.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>
#include <utility>

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

// Launch `kern` on stream `s` and report this launch's own outcome: the value
// cudaLaunchKernelEx returns, not the process-wide last-error state, which may
// hold an earlier, unrelated error that belongs to the caller (reading it with
// cudaGetLastError would also clear it).
template <typename... KArgs, typename... Args>
inline fp8q_status launch_on(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...) == cudaSuccess
             ? FP8Q_OK
             : FP8Q_ERR_CUDA;
}

// Time limit of every device-side wait (fp8q_set_wait_timeout_ns).
inline std::atomic<uint64_t> &wait_timeout_ns() {
  static std::atomic<uint64_t> ns{2000000000ull};
  return ns;
}

// The driver's tensor-map encoder, looked up through the runtime (no libcuda
// link dependency).
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// 2-D tensor [rows][cols] of `type` (elem_bytes each) with row pitch ld_bytes,
// box box_cols x box_rows, zero fill outside the tensor.
inline bool make_tmap_2d(CUtensorMap *m, CUtensorMapDataType type, const void *base,
                         uint64_t rows, uint64_t cols, uint64_t ld_bytes, uint32_t box_cols,
                         uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, type, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Read (and clear) the quantisers' device status word; defined in quant.cu.
fp8q_status quant_status_take(cudaStream_t s);
// The same for the power-of-two (block-scaled MMA) GEMM; defined in gemm_mx.cu.
fp8q_status mx_status_take(cudaStream_t s);

}  // namespace fp8q
