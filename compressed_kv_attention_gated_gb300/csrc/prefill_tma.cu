// prefill_tma.cu -- compress pass of the online c128 prefill, TMA-pipelined.
//
// Source: sglang page "sgl-project--sglang/.../deepseek_v4/c128_online.cuh"
// (flash_c128_online_prefill with kWrite = false, c128_prefill_forward): per
// compress segment and channel, a softmax over the segment's tokens with the
// chunk-position bias, merged with the slot's stored partial (max, sum, kv)
// when the segment starts mid-chunk; the kv of the merged softmax is written
// to the output row of the segment's last token.
//
// Design for sm_103a (memory bound; no dense contraction, no tensor cores):
//   * persistent: one CTA per SM, each owning a fixed 128-channel slice of
//     the row for all the segments it is given (plan p, p + G, p + 2G, ...);
//   * the slice of the bias table, pre-multiplied by log2(e), is staged in
//     shared memory once per CTA (128 x slice fp32);
//   * warp 0 is the producer: one lane walks the same segment sequence and
//     streams each segment as 64-row (bf16) or 32-row (fp32) boxes of kv and
//     of score with 2-D tiled
//     TMA loads (cp.async.bulk.tensor) into a ring of stages guarded by
//     full/empty mbarriers; rows past the input are zero-filled by the TMA
//     unit and masked by the consumers;
//   * the other warps (8 for bf16, 4 for fp32) are consumers: warp w reduces
//     rows [8w, 8w+8) of every stage
//     two-pass in registers (one ex2 per element, log2 domain), keeping a
//     running (max, sum, weighted sum) per channel; at the end of a segment the
//     eight partials meet in shared memory (double-buffered, mbarrier
//     synchronised), are merged with the prefetched prior state and stored.
//   * with the FP8 stage (kFp8) one more warp takes each segment's staged row
//     slice through the pooled path's rotation and quantisation into the
//     paged FP8 cache, joining the segment barrier two segments ahead once it
//     has read a row buffer, so the consumers never wait for it;
//   * every wait is bounded (two seconds of wall time); a timeout sets
//     CKV_DEVERR_TIMEOUT in the error word and the thread leaves; the producer
//     drains its own outstanding TMA loads before it exits.
#include <cudaTypedefs.h>

#include <mutex>

#include "ckv_device.cuh"
#include "ckv_fp8.cuh"
#include "ckv_launch.h"
#include "ckv_launch_util.cuh"
#include "ckv_tma.cuh"

namespace ckv {
namespace {

// Per input type: channels per slice (kCh), channels per consumer lane (kCpl),
// pipeline stages, consumer warps and rows per stage (the TMA box height; each
// consumer warp owns 8 rows of every stage).  A stage holds one box of kv and
// one of score, 16 KB each.
template <typename InT>
struct TmaCfg;
template <>
struct TmaCfg<float> {
  static constexpr int kCh = 128;     // 512 B of a row
  static constexpr int kCpl = 4;
  static constexpr int kStages = 4;
  static constexpr int kCWarps = 4;
  static constexpr int kRows = 32;
  static constexpr CUtensorMapDataType kType = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
};
template <>
struct TmaCfg<__nv_bfloat16> {
  static constexpr int kCh = 128;     // 256 B of a row
  static constexpr int kCpl = 4;
  static constexpr int kStages = 4;
  static constexpr int kCWarps = 8;
  static constexpr int kRows = 64;
  static constexpr CUtensorMapDataType kType = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
};

constexpr int kRowsPerWarp = 8;

template <typename InT, bool kFp8 = false>
struct Layout {
  static constexpr int kCh = TmaCfg<InT>::kCh, kSt = TmaCfg<InT>::kStages;
  static constexpr int kCWarps = TmaCfg<InT>::kCWarps, kRows = TmaCfg<InT>::kRows;
  static constexpr int kRowBytes = kCh * static_cast<int>(sizeof(InT));
  static constexpr int kBoxBytes = kRows * kRowBytes;                 // one array, one stage
  static constexpr int kThreads = (kCWarps + 1 + (kFp8 ? 1 : 0)) * 32;  // + producer (+ FP8 warp)
  static constexpr int kKv = 0;
  static constexpr int kSc = kKv + kSt * kBoxBytes;
  static constexpr int kApe = kSc + kSt * kBoxBytes;                  // [128][kCh] fp32 * log2(e)
  static constexpr int kPart = kApe + 128 * kCh * 4;                  // [2][kCWarps][3][kCh] fp32
  static constexpr int kRow = kPart + 2 * kCWarps * 3 * kCh * 4;     // FP8 stage: [2][kCh] fp32
  static constexpr int kBar = kRow + (kFp8 ? 2 * kCh * 4 : 0);       // full, empty, ready (, rowready)
  static constexpr int kBytes = kBar + (2 * kSt + 2 + (kFp8 ? 2 : 0)) * 8;
  // the FP8 warp reads one float4 per lane (128 channels) and stores it as one
  // 128-channel FP8 block per slice
  static_assert(!kFp8 || kCh == 128, "the FP8 warp stores one 128-channel block per slice");
  static_assert(kRows == kCWarps * kRowsPerWarp, "each consumer warp owns 8 rows of a stage");
};

struct Seg {
  uint32_t ragged, batch, pic, window;
  bool sentinel, ok;
};

__device__ __forceinline__ Seg decode_plan(const uint4 raw, const C128PrefillArgs& a) {
  Seg s;
  s.ragged = raw.x;
  s.batch = raw.y;
  s.pic = raw.z & 127u;
  s.window = raw.w;
  s.sentinel = raw.x == 0xFFFFFFFFu;
  s.ok = !s.sentinel && s.batch < static_cast<uint32_t>(a.B) && s.window >= 1 &&
         s.window <= s.pic + 1 && s.ragged < a.num_tokens && s.ragged + 1 >= s.window &&
         s.pic == 127u;
  return s;
}

__device__ __forceinline__ uint4 load_plan(const ckv_plan_entry* plan, uint32_t p, uint32_t n) {
  if (p >= n) return make_uint4(0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu);
  return *reinterpret_cast<const uint4*>(plan + p);
}

template <typename InT>
struct Row;  // kCpl channels of one smem row, widened to fp32
template <>
struct Row<float> {
  static __device__ __forceinline__ void load(const uint8_t* row, int lane, float (&v)[4]) {
    const float4 x = reinterpret_cast<const float4*>(row)[lane];
    v[0] = x.x;
    v[1] = x.y;
    v[2] = x.z;
    v[3] = x.w;
  }
};
template <>
struct Row<__nv_bfloat16> {
  static __device__ __forceinline__ void load(const uint8_t* row, int lane, float (&v)[4]) {
    const uint2 x = reinterpret_cast<const uint2*>(row)[lane];
    v[0] = bf16_lo(x.x);
    v[1] = bf16_hi(x.x);
    v[2] = bf16_lo(x.y);
    v[3] = bf16_hi(x.y);
  }
};

template <int kCpl>
__device__ __forceinline__ void load_ape(const float* ape_row, int lane, float (&v)[kCpl]) {
  if constexpr (kCpl == 2) {
    const float2 x = reinterpret_cast<const float2*>(ape_row)[lane];
    v[0] = x.x;
    v[1] = x.y;
  } else {
    const float4 x = reinterpret_cast<const float4*>(ape_row)[lane];
    v[0] = x.x;
    v[1] = x.y;
    v[2] = x.z;
    v[3] = x.w;
  }
}

template <int D, typename InT, bool kFp8>
__global__ void __launch_bounds__(Layout<InT, kFp8>::kThreads, 1)
    c128_prefill_tma_kernel(const __grid_constant__ CUtensorMap tmap,
                            const __grid_constant__ C128PrefillArgs a) {
  using L = Layout<InT, kFp8>;
  constexpr int kCh = TmaCfg<InT>::kCh, kCpl = TmaCfg<InT>::kCpl, kSt = TmaCfg<InT>::kStages;
  constexpr int kCWarps = L::kCWarps, kRows = L::kRows, kBoxBytes = L::kBoxBytes;
  constexpr int kThreads = L::kThreads, kRowBytes = L::kRowBytes;
  constexpr int S = D / kCh;
  extern __shared__ __align__(1024) uint8_t smem[];
  float* s_ape = reinterpret_cast<float*>(smem + L::kApe);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* empty = full + kSt;
  uint64_t* ready = empty + kSt;
  uint64_t* rowready = ready + 2;  // FP8 stage only: a segment's row is staged

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slice = blockIdx.x % S;
  const uint32_t group = blockIdx.x / S, ngroups = gridDim.x / S;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kSt; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kCWarps);
    }
    // with the FP8 stage the FP8 warp also arrives on `ready`: its arrival for
    // a segment means it has read the row buffer that segment will reuse
    mbar_init(&ready[0], kCWarps + (kFp8 ? 1 : 0));
    mbar_init(&ready[1], kCWarps + (kFp8 ? 1 : 0));
    if constexpr (kFp8) {
      mbar_init(&rowready[0], kCh / 32);
      mbar_init(&rowready[1], kCh / 32);
    }
    fence_mbar_init();
  }
  __syncthreads();  // barriers initialised before anyone waits on them
  pdl_wait();
  const uint32_t n = a.counts ? min(a.counts[0], a.num_compress) : a.num_compress;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // starts streaming at once: only the consumers need the bias slice
    pdl_trigger();
    if (lane != 0) return;
    uint32_t st = 0, ph = 0, armed = 0;
    bool aborted = false;
    uint4 next = load_plan(a.compress_plan, group, n);
    for (uint32_t p = group; p < n && !aborted; p += ngroups) {
      const uint4 cur = next;
      next = load_plan(a.compress_plan, p + ngroups, n);
      const Seg s = decode_plan(cur, a);
      if (!s.ok) continue;
      const int32_t first = static_cast<int32_t>(s.ragged - s.window + 1);
      const uint32_t nsub = (s.window + kRows - 1) / kRows;
      for (uint32_t k = 0; k < nsub; ++k) {
        if (!mbar_wait(&empty[st], ph ^ 1)) {
          flag_error(a.err, CKV_DEVERR_TIMEOUT);
          aborted = true;
          break;
        }
        mbar_arrive_expect_tx(&full[st], 2 * kBoxBytes);
        tma_load_2d(smem + L::kKv + st * kBoxBytes, &tmap, slice * kCh, first + k * kRows, &full[st]);
        tma_load_2d(smem + L::kSc + st * kBoxBytes, &tmap, D + slice * kCh, first + k * kRows, &full[st]);
        ++armed;
        if (++st == kSt) {
          st = 0;
          ph ^= 1;
        }
      }
    }
    // Leave no TMA load in flight: wait for the last arming of every stage.
    for (uint32_t x = 0; x < static_cast<uint32_t>(kSt); ++x) {
      if (armed > x && !mbar_wait(&full[x], x < st ? ph : (ph ^ 1))) flag_error(a.err, CKV_DEVERR_TIMEOUT);
    }
    return;
  }

  if constexpr (kFp8) {
    if (warp == kCWarps + 1) {
      // ---------------------------------------------------------- FP8 warp
      // takes each segment's staged row (block `slice` of the output row) and
      // stores it through the pooled output stage, while the consumers go on;
      // the consumers reuse a row buffer only after passing a `ready` barrier
      // that the FP8 warp joins once it has read that buffer
      pdl_trigger();
      if (lane == 0) {  // the first use of each row buffer needs no read to wait for
        mbar_arrive(&ready[0]);
        mbar_arrive(&ready[1]);
      }
      uint32_t it = 0;
      uint4 next = load_plan(a.compress_plan, group, n);
      for (uint32_t p = group; p < n; p += ngroups) {
        const uint4 cur = next;
        next = load_plan(a.compress_plan, p + ngroups, n);
        const Seg s = decode_plan(cur, a);
        if (!s.ok) continue;  // the consumers skip it too
        const int buf = static_cast<int>(it & 1);
        const uint32_t par = (it >> 1) & 1;
        ++it;
        bool slot_ok = true;
        if (s.pic + 1 != s.window) {
          const int32_t li = a.load_indices[s.batch];
          slot_ok = li >= 0 && li < a.num_slots;
        }
        const int64_t loc = a.cache_loc[s.ragged];
        if (!mbar_wait(&rowready[buf], par)) {
          if (lane == 0) flag_error(a.err, CKV_DEVERR_TIMEOUT);
          return;
        }
        const float4 v = reinterpret_cast<const float4*>(smem + L::kRow + buf * kCh * 4)[lane];
        __syncwarp();
        if (lane == 0) mbar_arrive(&ready[buf]);  // counts toward the segment two ahead
        if (!slot_ok) continue;
        if (loc < 0 || loc >= a.num_pages * a.page_size) {
          if (lane == 0 && slice == 0) flag_error(a.err, CKV_DEVERR_CACHE_LOC);
          continue;
        }
        const float x[4] = {v.x, v.y, v.z, v.w};
        float xb[4], yb[4], scale;
        uint32_t codes;
        if (a.round_scale) rotate_quantize<true>(x, lane, codes, scale, xb, yb);
        else rotate_quantize<false>(x, lane, codes, scale, xb, yb);
        cache_write_block(a.cache, a.page_size, loc, S, slice, lane, codes, scale);
      }
      return;
    }
  }

  // -------------------------------------------------------------- consumers
  // bias slice, pre-scaled to the log2 domain, staged by the consumer warps
  // (named barrier 1) while the producer's first loads are in flight
  for (int i = threadIdx.x - 32; i < 128 * kCh / 4; i += kCWarps * 32) {
    const int j = i / (kCh / 4), c4 = i % (kCh / 4);
    float4 v = ld_shared_ro_f4(a.ape + j * D + slice * kCh + 4 * c4);
    v.x *= kLog2e;
    v.y *= kLog2e;
    v.z *= kLog2e;
    v.w *= kLog2e;
    reinterpret_cast<float4*>(s_ape)[i] = v;
  }
  asm volatile("bar.sync 1, %0;" ::"r"(kCWarps * 32) : "memory");
  pdl_trigger();
  const int cw = warp - 1;
  const int t = cw * 32 + lane;  // channel of the slice in the epilogue (t < kCh)
  uint32_t st = 0, ph = 0, it = 0;
  uint4 next = load_plan(a.compress_plan, group, n);
  for (uint32_t p = group; p < n; p += ngroups) {
    const uint4 cur = next;
    next = load_plan(a.compress_plan, p + ngroups, n);
    const Seg s = decode_plan(cur, a);
    if (!s.ok) {
      if (!s.sentinel && t == 0) flag_error(a.err, CKV_DEVERR_PLAN);
      continue;
    }
    const int chunk_offset = static_cast<int>(s.pic + 1 - s.window);
    // stored partial of a segment that starts mid-chunk: fetched now, used at the end
    bool prior = chunk_offset != 0, slot_ok = true;
    float m1 = 0.f, s1 = 0.f, k1 = 0.f;
    if (prior) {
      const int32_t li = a.load_indices[s.batch];
      slot_ok = li >= 0 && li < a.num_slots;
      if (!slot_ok && t == 0) flag_error(a.err, CKV_DEVERR_SLOT);
      if (slot_ok && t < kCh) {
        const float* ld = a.state + static_cast<int64_t>(li) * 3 * D + slice * kCh + t;
        m1 = ld[0];
        s1 = ld[D];
        k1 = ld[2 * D];
      }
    }

    float M[kCpl], Sm[kCpl], A[kCpl];
#pragma unroll
    for (int c = 0; c < kCpl; ++c) {
      M[c] = kNegBig;
      Sm[c] = 0.f;
      A[c] = 0.f;
    }
    const uint32_t nsub = (s.window + kRows - 1) / kRows;
    for (uint32_t k = 0; k < nsub; ++k) {
      if (!mbar_wait(&full[st], ph)) {
        if (lane == 0) flag_error(a.err, CKV_DEVERR_TIMEOUT);
        return;
      }
      const int r0 = static_cast<int>(k) * kRows + cw * kRowsPerWarp;  // first row of this warp
      const int nvalid = min(kRowsPerWarp, max(0, static_cast<int>(s.window) - r0));
      if (nvalid > 0) {
        const uint8_t* kvb = smem + L::kKv + st * kBoxBytes + cw * kRowsPerWarp * kRowBytes;
        const uint8_t* scb = smem + L::kSc + st * kBoxBytes + cw * kRowsPerWarp * kRowBytes;
        const float* apb = s_ape + (chunk_offset + r0) * kCh;
        float z[kRowsPerWarp][kCpl], kv[kRowsPerWarp][kCpl];
        float bm[kCpl];
#pragma unroll
        for (int c = 0; c < kCpl; ++c) bm[c] = kNegBig;
        if (nvalid == kRowsPerWarp) {
#pragma unroll
          for (int r = 0; r < kRowsPerWarp; ++r) {
            float sc[kCpl], ap[kCpl];
            Row<InT>::load(kvb + r * kRowBytes, lane, kv[r]);
            Row<InT>::load(scb + r * kRowBytes, lane, sc);
            load_ape<kCpl>(apb + r * kCh, lane, ap);
#pragma unroll
            for (int c = 0; c < kCpl; ++c) {
              z[r][c] = fmaf(sc[c], kLog2e, ap[c]);
              bm[c] = fmaxf(bm[c], z[r][c]);
            }
          }
        } else {
#pragma unroll
          for (int r = 0; r < kRowsPerWarp; ++r) {
            if (r < nvalid) {
              float sc[kCpl], ap[kCpl];
              Row<InT>::load(kvb + r * kRowBytes, lane, kv[r]);
              Row<InT>::load(scb + r * kRowBytes, lane, sc);
              load_ape<kCpl>(apb + r * kCh, lane, ap);
#pragma unroll
              for (int c = 0; c < kCpl; ++c) {
                z[r][c] = fmaf(sc[c], kLog2e, ap[c]);
                bm[c] = fmaxf(bm[c], z[r][c]);
              }
            } else {
#pragma unroll
              for (int c = 0; c < kCpl; ++c) {
                z[r][c] = kNegBig;  // weight ex2(kNegBig - bm) == 0
                kv[r][c] = 0.f;
              }
            }
          }
        }
#pragma unroll
        for (int c = 0; c < kCpl; ++c) {
          float bs = 0.f, ba = 0.f;
#pragma unroll
          for (int r = 0; r < kRowsPerWarp; ++r) {
            const float e = fast_exp2(z[r][c] - bm[c]);
            bs += e;
            ba = fmaf(e, kv[r][c], ba);
          }
          const float nm = fmaxf(M[c], bm[c]);
          const float f1 = fast_exp2(M[c] - nm), f2 = fast_exp2(bm[c] - nm);
          Sm[c] = Sm[c] * f1 + bs * f2;
          A[c] = A[c] * f1 + ba * f2;
          M[c] = nm;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      if (++st == kSt) {
        st = 0;
        ph ^= 1;
      }
    }

    // merge the eight warp partials of this segment (double-buffered by segment parity)
    const int buf = it & 1;
    float* part = reinterpret_cast<float*>(smem + L::kPart) + buf * kCWarps * 3 * kCh;
#pragma unroll
    for (int c = 0; c < kCpl; ++c) {
      part[(cw * 3 + 0) * kCh + lane * kCpl + c] = M[c];
      part[(cw * 3 + 1) * kCh + lane * kCpl + c] = Sm[c];
      part[(cw * 3 + 2) * kCh + lane * kCpl + c] = A[c];
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&ready[buf]);
    const uint32_t seg_parity = (it >> 1) & 1;
    if (!mbar_wait(&ready[buf], seg_parity)) {
      if (lane == 0) flag_error(a.err, CKV_DEVERR_TIMEOUT);
      return;
    }
    ++it;
    if (t < kCh && slot_ok) {
      float m = kNegBig;
#pragma unroll
      for (int w = 0; w < kCWarps; ++w) m = fmaxf(m, part[(w * 3) * kCh + t]);
      float ssum = 0.f, acc = 0.f;
#pragma unroll
      for (int w = 0; w < kCWarps; ++w) {
        const float f = fast_exp2(part[(w * 3) * kCh + t] - m);
        ssum = fmaf(part[(w * 3 + 1) * kCh + t], f, ssum);
        acc = fmaf(part[(w * 3 + 2) * kCh + t], f, acc);
      }
      float kvout = acc / ssum;
      if (prior) {
        const float m1l = m1 * kLog2e;
        const float nm = fmaxf(m1l, m);
        const float w1 = s1 * fast_exp2(m1l - nm), w2 = ssum * fast_exp2(m - nm);
        kvout = (k1 * w1 + kvout * w2) / (w1 + w2);
      }
      if (a.out) a.out[static_cast<int64_t>(s.ragged) * D + slice * kCh + t] = kvout;
      if constexpr (kFp8) reinterpret_cast<float*>(smem + L::kRow)[buf * kCh + t] = kvout;
    }
    if constexpr (kFp8) {
      // the epilogue warps hand the row slice to the FP8 warp
      if (cw < kCh / 32) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&rowready[buf]);
      }
    }
  }
}

// A wait that nothing will ever satisfy: one thread arms an mbarrier for one
// arrival that never comes and waits on it with the given limit; the bounded
// wait must give up, flag CKV_DEVERR_TIMEOUT and return.
__global__ void wait_timeout_selftest_kernel(int32_t* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  if (!mbar_wait(&bar, 0, limit_ns)) flag_error(err, CKV_DEVERR_TIMEOUT);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

template <int D, typename InT, bool kFp8>
cudaError_t launch_grid(const CUtensorMap& map, const C128PrefillArgs& a, int sms, bool use_pdl, cudaStream_t s);

template <int D, typename InT>
cudaError_t launch_d(const C128PrefillArgs& a, bool use_pdl, cudaStream_t s) {
  using Cfg = TmaCfg<InT>;
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  CUtensorMap map;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(2 * D), static_cast<cuuint64_t>(a.num_tokens)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(2 * D * sizeof(InT))};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(Cfg::kCh), static_cast<cuuint32_t>(Cfg::kRows)};
  const cuuint32_t estr[2] = {1, 1};
  if (fn(&map, Cfg::kType, 2, const_cast<void*>(a.input), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorNotSupported;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (a.cache) return launch_grid<D, InT, true>(map, a, sms, use_pdl, s);
  return launch_grid<D, InT, false>(map, a, sms, use_pdl, s);
}

template <int D, typename InT, bool kFp8>
cudaError_t launch_grid(const CUtensorMap& map, const C128PrefillArgs& a, int sms, bool use_pdl, cudaStream_t s) {
  using L = Layout<InT, kFp8>;
  constexpr int S = D / TmaCfg<InT>::kCh;
  auto kern = c128_prefill_tma_kernel<D, InT, kFp8>;
  cudaError_t e = set_max_smem_once<c128_prefill_tma_kernel<D, InT, kFp8>>(L::kBytes);
  if (e != cudaSuccess) return e;
  const int grid = sms >= S ? (sms / S) * S : S;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(L::kThreads);
  cfg.dynamicSmemBytes = L::kBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = use_pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, map, a);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(int32_t* err, uint64_t limit_ns, cudaStream_t s) {
  return launch_ex(wait_timeout_selftest_kernel, dim3(1), dim3(32), 0, false, s, err, limit_ns);
}

bool c128_prefill_tma_supported(const C128PrefillArgs& a, int D, int in_dtype) {
  (void)D;
  (void)in_dtype;
  // TMA needs a 16-byte aligned base (checked by the C ABI), a row stride that
  // is a multiple of 16 bytes (2D * element size: always) and int32 row
  // coordinates.
  return a.num_tokens > 0 && a.num_tokens < (1ll << 31) && encode_fn() != nullptr;
}

cudaError_t launch_c128_prefill_compress_tma(const C128PrefillArgs& a, int D, int in_dtype,
                                             bool use_pdl, cudaStream_t s) {
  if (in_dtype == CKV_F32) {
    if (D == 128) return launch_d<128, float>(a, use_pdl, s);
    if (D == 256) return launch_d<256, float>(a, use_pdl, s);
    if (D == 512) return launch_d<512, float>(a, use_pdl, s);
  } else {
    if (D == 128) return launch_d<128, __nv_bfloat16>(a, use_pdl, s);
    if (D == 256) return launch_d<256, __nv_bfloat16>(a, use_pdl, s);
    if (D == 512) return launch_d<512, __nv_bfloat16>(a, use_pdl, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace ckv
