// planner_device.cu -- the online c128 prefill planner as a CUDA kernel.
//
// Same output as the host planner (sglang page "deepseek_v4/c128_online.cuh",
// plan_online_prefill_host), computed on the device so that planning and the
// prefill launches can be enqueued (or captured in a CUDA graph) without a
// host round trip.  Request b covers positions [prefix_b, seq_b), prefix_b =
// seq_b - extend_b; it owns
//   nc_b = seq_b / 128 - prefix_b / 128      compress segments (chunk ends
//                                            127, 255, ... inside the range)
//   nw_b = (seq_b % 128 != 0)                write segment (the trailing part)
// and the ragged rows after those of requests 0..b-1.
//
// Every CTA scans the request lengths itself (exclusive prefix sums of nc, nw
// and extend in shared memory), so no global scratch and no second launch are
// needed; then the grid writes entries in parallel, each thread finding its
// request by binary search over the prefix sums.  Invalid lengths set
// CKV_DEVERR_PLAN and make both counts 0.
#include <cstdint>

#include "ckv_device.cuh"
#include "ckv_launch.h"
#include "ckv_launch_util.cuh"

namespace ckv {
namespace {

constexpr int kPlanThreads = 1024;

struct PlanDevArgs {
  const int64_t* seq_lens;
  const int64_t* extend_lens;
  ckv_plan_entry* compress_plan;
  ckv_plan_entry* write_plan;
  uint32_t* counts;
  int32_t* err;
  uint32_t B;
  uint32_t num_tokens;
  int32_t pad;
};

// Block-wide exclusive scan of one value per thread (kPlanThreads threads).
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* s_warp, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = s_warp[lane];  // kPlanThreads / 32 == 32 warps
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;  // inclusive warp totals
  }
  __syncthreads();
  const uint32_t before = (warp > 0 ? s_warp[warp - 1] : 0u) + x - v;
  total = s_warp[31];
  __syncthreads();
  return before;
}

// Largest b in [0, B) with pre[b] <= e (pre is non-decreasing, pre[0] = 0).
__device__ __forceinline__ uint32_t find_request(const uint32_t* pre, uint32_t B, uint32_t e) {
  uint32_t lo = 0, hi = B - 1;
  while (lo < hi) {
    const uint32_t mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= e) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kPlanThreads) plan_device_kernel(const __grid_constant__ PlanDevArgs a) {
  extern __shared__ __align__(16) uint32_t s_plan[];
  uint32_t* s_c = s_plan;             // exclusive prefix of compress counts [B]
  uint32_t* s_w = s_c + a.B;          // exclusive prefix of write counts [B]
  uint32_t* s_r = s_w + a.B;          // ragged base [B]
  uint32_t* s_pre = s_r + a.B;        // prefix length [B]
  uint32_t* s_seq = s_pre + a.B;      // sequence length [B]
  __shared__ uint32_t s_warp[32];
  __shared__ uint32_t s_bad;

  pdl_wait();
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  uint32_t carry_c = 0, carry_w = 0, carry_r = 0;
  for (uint32_t base = 0; base < a.B; base += kPlanThreads) {
    const uint32_t b = base + threadIdx.x;
    uint32_t nc = 0, nw = 0, ext = 0;
    if (b < a.B) {
      const int64_t seq = a.seq_lens[b], e = a.extend_lens[b];
      if (e <= 0 || e > seq || seq > static_cast<int64_t>(UINT32_MAX)) {
        atomicOr(&s_bad, 1u);
      } else {
        const uint32_t s32 = static_cast<uint32_t>(seq), p32 = static_cast<uint32_t>(seq - e);
        nc = s32 / 128u - p32 / 128u;
        nw = (s32 % 128u) != 0u;
        ext = static_cast<uint32_t>(e);
        s_pre[b] = p32;
        s_seq[b] = s32;
      }
    }
    uint32_t tc, tw, tr;
    const uint32_t oc = block_exclusive_scan(nc, s_warp, tc);
    const uint32_t ow = block_exclusive_scan(nw, s_warp, tw);
    const uint32_t orr = block_exclusive_scan(ext, s_warp, tr);
    if (b < a.B) {
      s_c[b] = carry_c + oc;
      s_w[b] = carry_w + ow;
      s_r[b] = carry_r + orr;
    }
    carry_c += tc;
    carry_w += tw;
    carry_r += tr;
  }
  __syncthreads();
  const uint32_t NC = carry_c, NW = carry_w;
  if (s_bad || carry_r != a.num_tokens) {
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      flag_error(a.err, CKV_DEVERR_PLAN);
      a.counts[0] = 0;
      a.counts[1] = 0;
    }
    return;
  }
  const uint32_t limit_c = a.pad ? a.num_tokens : NC;
  const uint32_t limit_w = a.pad ? a.num_tokens : NW;
  const uint32_t stride = gridDim.x * blockDim.x;
  const uint4 sentinel = make_uint4(0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu);
  for (uint32_t e = blockIdx.x * blockDim.x + threadIdx.x; e < limit_c; e += stride) {
    uint4 v = sentinel;
    if (e < NC) {
      const uint32_t b = find_request(s_c, a.B, e);
      const uint32_t chunk = s_pre[b] / 128u + (e - s_c[b]);
      const uint32_t last = chunk * 128u + 127u;
      const uint32_t first = max(s_pre[b], chunk * 128u);
      v = make_uint4(s_r[b] + (last - s_pre[b]), b, last, last - first + 1u);
    }
    reinterpret_cast<uint4*>(a.compress_plan)[e] = v;
  }
  for (uint32_t e = blockIdx.x * blockDim.x + threadIdx.x; e < limit_w; e += stride) {
    uint4 v = sentinel;
    if (e < NW) {
      const uint32_t b = find_request(s_w, a.B, e);
      const uint32_t last = s_seq[b] - 1u;
      const uint32_t first = max(s_pre[b], (last / 128u) * 128u);
      v = make_uint4(s_r[b] + (last - s_pre[b]), b, last, last - first + 1u);
    }
    reinterpret_cast<uint4*>(a.write_plan)[e] = v;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    a.counts[0] = limit_c;
    a.counts[1] = limit_w;
  }
}

}  // namespace

cudaError_t launch_plan_device(const int64_t* seq_lens, const int64_t* extend_lens, uint32_t B,
                               uint32_t num_tokens, ckv_plan_entry* compress_plan,
                               ckv_plan_entry* write_plan, bool pad, uint32_t* counts,
                               int32_t* err, bool use_pdl, cudaStream_t s) {
  PlanDevArgs a;
  a.seq_lens = seq_lens;
  a.extend_lens = extend_lens;
  a.compress_plan = compress_plan;
  a.write_plan = write_plan;
  a.counts = counts;
  a.err = err;
  a.B = B;
  a.num_tokens = num_tokens;
  a.pad = pad ? 1 : 0;
  const size_t smem = static_cast<size_t>(B) * 5 * sizeof(uint32_t);
  // sized for the largest B the entry point accepts (8192 requests, 160 KB)
  cudaError_t e = set_max_smem_once<plan_device_kernel>(8192 * 5 * sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  // entries to write: at most num_tokens / 128 + B compress and B write segments
  // (or num_tokens of each with padding)
  const uint64_t work = pad ? num_tokens : static_cast<uint64_t>(num_tokens) / 128u + B;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const uint64_t want = (work + kPlanThreads - 1) / kPlanThreads;
  const unsigned grid = static_cast<unsigned>(want < 1 ? 1 : (want > static_cast<uint64_t>(sms) ? sms : want));
  return launch_ex(plan_device_kernel, dim3(grid), dim3(kPlanThreads), smem, use_pdl, s, a);
}

}  // namespace ckv
