// validate.cu -- debug check of the caller contract the compression kernels
// rely on: within one call the ids of a kind (state slots, cache locations,
// tail blocks) are distinct.  No counterpart in the sources, which state the
// contract and leave it unchecked.
//
// A bitmap of `range` bits in caller-provided scratch: one kernel clears it,
// a second one sets the bit of every non-negative id with atomicOr and flags
// CKV_DEVERR_DISTINCT when the bit was set already (a repeat) or the id is
// out of range.  Both kernels are grid-stride loops over a grid of a few CTAs
// per SM.
#include <cstdint>

#include "ckv_device.cuh"
#include "ckv_launch.h"
#include "ckv_launch_util.cuh"

namespace ckv {
namespace {

constexpr int kCheckThreads = 256;

__global__ void __launch_bounds__(kCheckThreads) clear_bits_kernel(uint32_t* bits, int64_t words) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < words; i += stride)
    bits[i] = 0u;
}

template <typename Id>
__global__ void __launch_bounds__(kCheckThreads)
    mark_distinct_kernel(const Id* ids, int64_t n, int64_t range, uint32_t* bits, int32_t* err) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int64_t id = static_cast<int64_t>(ids[i]);
    if (id < 0) continue;  // padding
    if (id >= range) {
      flag_error(err, CKV_DEVERR_DISTINCT);
      continue;
    }
    const uint32_t m = 1u << (id & 31);
    if (atomicOr(bits + (id >> 5), m) & m) flag_error(err, CKV_DEVERR_DISTINCT);
  }
}

unsigned grid_for(int64_t work, int sms) {
  const int64_t want = (work + kCheckThreads - 1) / kCheckThreads;
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  return static_cast<unsigned>(want < 1 ? 1 : (want > cap ? cap : want));
}

}  // namespace

cudaError_t launch_check_distinct(const void* ids, int id_bytes, int64_t n, int64_t range, uint32_t* bits,
                                  int32_t* err, cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int64_t words = (range + 31) / 32;
  e = launch_ex(clear_bits_kernel, dim3(grid_for(words, sms)), dim3(kCheckThreads), 0, false, s, bits, words);
  if (e != cudaSuccess || n == 0) return e;
  if (id_bytes == 4)
    return launch_ex(mark_distinct_kernel<int32_t>, dim3(grid_for(n, sms)), dim3(kCheckThreads), 0, false, s,
                     static_cast<const int32_t*>(ids), n, range, bits, err);
  return launch_ex(mark_distinct_kernel<int64_t>, dim3(grid_for(n, sms)), dim3(kCheckThreads), 0, false, s,
                   static_cast<const int64_t*>(ids), n, range, bits, err);
}

}  // namespace ckv
