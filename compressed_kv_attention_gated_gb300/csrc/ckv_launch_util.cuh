// ckv_launch_util.cuh -- kernel launch with an optional programmatic dependency.
#pragma once

#include <cuda_runtime.h>

namespace ckv {

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
