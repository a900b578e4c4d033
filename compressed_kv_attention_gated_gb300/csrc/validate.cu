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
#include <mutex>

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

// ---------------------------------------------------------------------------
// Allocation-free variant.  Some callers cannot hand the check a scratch
// buffer: a serving engine that reserves nearly all HBM for its paged KV cache
// and owns every byte of it through its own allocator, or a loop that must not
// call cudaMalloc because cudaMalloc may synchronise the device and stall it.
// For them the bitmap lives in this file-scope array, which every GPU that
// loads the library holds until the process exits; every call shares it.  In
// host code `g_noalloc_bits` is only a host-side stand-in for the symbol, never
// a device address: the device address is looked up with cudaGetSymbolAddress,
// once per device, with that device current.
constexpr int64_t kNoAllocWords = int64_t{1} << 16;  // 256 KB: ids in [0, 2^21)
static __device__ __align__(256) uint32_t g_noalloc_bits[kNoAllocWords];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
uint32_t* g_noalloc_ptr[kMaxDevices] = {};
}  // namespace

int64_t noalloc_check_max_range() { return kNoAllocWords * 32; }

cudaError_t launch_check_distinct_noalloc(const void* ids, int id_bytes, int64_t n, int64_t range, int32_t* err,
                                          cudaStream_t s) {
  if (range > kNoAllocWords * 32) return cudaErrorInvalidValue;  // the entry point rejects this first
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  uint32_t* bits = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_bits);
      if (e != cudaSuccess) return e;
      g_noalloc_ptr[dev] = static_cast<uint32_t*>(p);
    }
    bits = g_noalloc_ptr[dev];
  }
  // the clear kernel resets the words this call uses before any id is marked
  return launch_check_distinct(ids, id_bytes, n, range, bits, err, s);
}

}  // namespace ckv
