// probe.cu -- latency floors of a decode-sized launch (a measurement aid).
//
// The pooled decode update is bound by latency, not bandwidth: one call moves
// about 3 MB, and a closing pool needs two dependent global round trips (its
// token's index words, then the ring rows they name).  These kernels take a
// decode kernel's launch shape (n warps, a chosen number per CTA) and do
// nothing but the dependent memory traffic of that critical path, so that
// timing them with the same method as the decode call gives its floor:
//   hops 0  wait for the predecessor grid (programmatic dependent launch) and
//           return: the launch-and-completion cost alone;
//   hops 1  each warp loads the 4-byte word idx[w] and lane 0 stores it: one
//           global round trip;
//   hops 2  each warp loads idx[w], then the 256-byte row rows[idx[w]] (8 bytes
//           per lane), then stores that row: two dependent round trips.
//   hops 3  one round trip carrying the pooled decode's first-hop loads: each
//           thread loads 12 index words (idx[b0 .. b0 + 15], the same for the
//           warp, b0 = w rounded down to a multiple of 4 and kept inside idx)
//           and 8 four-byte row words 256 bytes apart, and lane 0 stores the
//           exclusive or of the 20 words it loaded.
//   hops 4  the pooled decode's memory pattern without its arithmetic: the
//           first hop of hops 3, except that each warp pair (a request)
//           reads 8 rows of its own, each warp one half of each; then, for
//           one warp pair in four (a request whose pool closes), a second hop
//           that depends on idx[w]: 30 row words per thread from the 8 KB
//           block holding row idx[w] (as a closing pool's 15 key and 15 score
//           ring rows), issued before each thread stores its 8 first-hop row
//           words (1 KB per warp, as the ring stashes of a request's tokens);
//           lane 0 finally stores the exclusive or of all it loaded.  The
//           grid's dependents are released after the first hop, as in the
//           decode.
// Every load takes the read-only path (ld.global.nc), as the decode's own
// index and row loads do.  An index outside [0, num_rows) is skipped.
#include <cstdint>

#include "ckv_device.cuh"
#include "ckv_launch_util.cuh"

namespace ckv {
namespace {

// x mod m for x >= 0, m > 0, with no division when x < m already (a 64-bit
// division would add its own latency in front of the loads being measured)
__device__ __forceinline__ int64_t wrap(int64_t x, int64_t m) { return x < m ? x : x % m; }

template <int kHops>
__global__ void latency_probe_kernel(const int32_t* idx, const uint2* rows, int64_t num_rows, uint2* out,
                                     int32_t n_warps) {
  pdl_wait();
  if constexpr (kHops != 4) pdl_trigger();
  if constexpr (kHops > 0) {
    const int lane = threadIdx.x & 31;
    const int64_t w = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (w >= n_warps) return;
    const int32_t r = __ldg(idx + w);
    if constexpr (kHops == 1) {
      if (lane == 0) reinterpret_cast<int32_t*>(out + w * 32)[0] = r;
    } else if constexpr (kHops == 2) {
      if (r < 0 || r >= num_rows) return;
      out[w * 32 + lane] = __ldg(rows + static_cast<int64_t>(r) * 32 + lane);
    } else if constexpr (kHops == 3) {
      // n_warps >= 16 and num_rows >= 9 (checked by the caller): the 16 index
      // words and the 8 row words below stay inside idx and rows
      const int64_t b0 = min(w & ~int64_t{3}, static_cast<int64_t>(n_warps) - 16);
      int32_t acc = r;
#pragma unroll
      for (int q = 1; q < 12; ++q) acc ^= __ldg(idx + b0 + ((q * 7) & 15));
      const uint32_t* rw = reinterpret_cast<const uint32_t*>(rows) + wrap(w * 8, num_rows * 64 - 512) + lane;
#pragma unroll
      for (int q = 0; q < 8; ++q) acc ^= static_cast<int32_t>(__ldg(rw + q * 64));
      if (lane == 0) reinterpret_cast<int32_t*>(out + w * 32)[0] = acc;
    } else {
      // n_warps >= 16 and num_rows >= 64 (checked by the caller); out holds
      // 1 KB per warp
      const int64_t b0 = min(w & ~int64_t{3}, static_cast<int64_t>(n_warps) - 16);
      int32_t acc = r;
#pragma unroll
      for (int q = 1; q < 12; ++q) acc ^= __ldg(idx + b0 + ((q * 7) & 15));
      // each warp pair (a request) reads its own 2 KB: 8 rows, a half-row each warp
      const uint32_t* rw = reinterpret_cast<const uint32_t*>(rows) + wrap((w >> 1) * 512, num_rows * 64 - 512) +
                           (w & 1) * 32 + lane;
      uint32_t v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = __ldg(rw + q * 64);
      pdl_trigger();
      const bool closing = ((w >> 1) & 3) == 0 && r >= 0 && r < num_rows;
      uint32_t hv[30];
      if (closing) {
        // the 8 KB block of 32 rows holding row r (the last whole block past it)
        const int64_t b = min(static_cast<int64_t>(r >> 5), num_rows / 32 - 1);
        const uint32_t* blk = reinterpret_cast<const uint32_t*>(rows) + b * 2048 + (w & 1) * 32 + lane;
#pragma unroll
        for (int q = 0; q < 15; ++q) {
          hv[q] = __ldg(blk + q * 64);
          hv[15 + q] = __ldg(blk + (16 + q) * 64);
        }
      }
      uint32_t* o = reinterpret_cast<uint32_t*>(out) + w * 256 + lane;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        o[q * 32] = v[q];
        acc ^= static_cast<int32_t>(v[q]);
      }
      if (closing) {
#pragma unroll
        for (int q = 0; q < 30; ++q) acc ^= static_cast<int32_t>(hv[q]);
      }
      if (lane == 0) reinterpret_cast<int32_t*>(out)[w * 256] = acc;
    }
  }
}

}  // namespace

cudaError_t launch_latency_probe(int hops, const int32_t* idx, const void* rows, int64_t num_rows, void* out,
                                 int32_t n_warps, int32_t warps_per_cta, bool use_pdl, cudaStream_t s) {
  const unsigned ctas = static_cast<unsigned>((n_warps + warps_per_cta - 1) / warps_per_cta);
  const dim3 grid(ctas > 0 ? ctas : 1u), block(32 * warps_per_cta);
  const uint2* r = static_cast<const uint2*>(rows);
  uint2* o = static_cast<uint2*>(out);
  switch (hops) {
    case 0: return launch_ex(latency_probe_kernel<0>, grid, block, 0, use_pdl, s, idx, r, num_rows, o, n_warps);
    case 1: return launch_ex(latency_probe_kernel<1>, grid, block, 0, use_pdl, s, idx, r, num_rows, o, n_warps);
    case 2: return launch_ex(latency_probe_kernel<2>, grid, block, 0, use_pdl, s, idx, r, num_rows, o, n_warps);
    case 3: return launch_ex(latency_probe_kernel<3>, grid, block, 0, use_pdl, s, idx, r, num_rows, o, n_warps);
    case 4: return launch_ex(latency_probe_kernel<4>, grid, block, 0, use_pdl, s, idx, r, num_rows, o, n_warps);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ckv
