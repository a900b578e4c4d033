// ckv_launch_util.cuh -- kernel launch with an optional programmatic dependency.
#pragma once

#include <atomic>
#include <cstdint>

#include <cuda_runtime.h>

namespace ckv {

// Raise the dynamic shared-memory limit of kernel Kern on the current device,
// once per device (so that later launches, e.g. inside a stream capture, make
// no attribute calls).
template <auto Kern>
cudaError_t set_max_smem_once(int bytes) {
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Launch `k` on stream `s`; with use_pdl the launch may begin before the
// preceding grid in the stream finishes (the kernel itself must execute
// griddepcontrol.wait before touching memory that grid may write).
template <typename... Args>
cudaError_t launch_ex(void (*k)(Args...), dim3 grid, dim3 block, size_t smem, bool use_pdl,
                      cudaStream_t s, const Args&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = use_pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, args...);
}

}  // namespace ckv
