// c128.cu -- online P=128 gated-softmax compression (decode and prefill).
//
// Source: sglang page "sgl-project--sglang/.../deepseek_v4/c128_online.cuh"
// (flash_c128_online_decode, c128_prefill_forward, flash_c128_online_prefill,
// run_decode, run_prefill).  State layout per slot: fp32 [3][D] = max | sum | kv
// with kv normalised; input row: [2D] = kv | score.
//
// Design for sm_103a (memory bound, SIMT, no tensor cores):
//   decode  -- two 4-channel groups per thread (D / 8 threads per request,
//              the whole batch resident in one wave); the input row is issued
//              before the slot index is known, the slot state is skipped at
//              chunk position 0, unchanged 32-byte sectors of the running max
//              are not rewritten; two ex2 per channel.
//   prefill -- one CTA of 8 warps per (segment, 128-channel slice).  Warp w
//              owns chunk positions [16w, 16w+16), loads them 8 tokens at a
//              time (16-byte fp32 / 8-byte bf16 vectors, streaming hints) and
//              reduces them two-pass in registers (one ex2 per element); the 8
//              warp partials (max, sum, weighted sum) are merged through shared
//              memory, then merged with the stored partial state when the
//              segment starts mid-chunk, then stored.  Compress and write
//              passes are two launches in stream order (optionally chained
//              by programmatic dependent launch).
//   FP8 stage (the _fp8 calls; kFp8 instantiations) -- each emitted row is
//              stored, 128-channel block by block, through the pooled path's
//              rotation and quantisation (ckv_fp8.cuh) into a paged FP8
//              cache.  The decode at D >= 256 rotates straight from the
//              closing request's registers (its threads already hold each
//              block in the rotation's lane layout); the decode at D = 128
//              and the prefill stage the row in shared memory first.
#include <type_traits>

#include "ckv_device.cuh"
#include "ckv_fp8.cuh"
#include "ckv_launch.h"
#include "ckv_launch_util.cuh"

namespace ckv {
namespace {

// --------------------------------------------------------------------------
// decode
// --------------------------------------------------------------------------
constexpr int kDecodeThreads = 256;
constexpr int kDecodeGroups = 2;     // float4 channel groups per thread
constexpr int kDecodeMinBlocks = 4;  // CTAs per SM (64 registers, no spills)
constexpr int kDecodeFp8MinBlocks = 4;  // with the FP8 output stage

// Thread t of a request owns G groups of 4 channels, 4t + (D / G) g: D / (4G)
// threads per request and 256 / (D / (4G)) requests per CTA, so the whole
// decode batch is resident at once and every request's loads are in flight
// together.
// Row marker of the FP8 output stage: this request emits no row.
constexpr int64_t kNoRow = INT64_MIN;

template <int D, typename InT, int G, int kMinBlocks, bool kFp8>
__global__ void __launch_bounds__(kDecodeThreads, kMinBlocks)
    c128_decode_kernel(const __grid_constant__ C128DecodeArgs a) {
  constexpr int kTpr = D / (4 * G);             // threads per request (even)
  constexpr int kRpc = kDecodeThreads / kTpr;   // requests per CTA
  constexpr int kSpan = D / G;                  // channel distance between groups
  // FP8 stage straight from registers when a request is whole warps and each
  // group spans whole 128-channel blocks (D >= 256 with two groups)
  constexpr bool kWarpRows = kTpr % 32 == 0 && kSpan % 128 == 0;
  pdl_wait();
  pdl_trigger();
  const int t = threadIdx.x % kTpr;
  const int b = blockIdx.x * kRpc + threadIdx.x / kTpr;
  // no early return: lane pairs exchange a flag at the end
  const bool in_batch = b < a.B;

  // The slot index gates the dependent state loads: issue it before the input stream.
  const int32_t index = in_batch ? a.indices[b] : 0;
  const int32_t seq_len = in_batch ? a.seq_lens[b] : 1;
  // the FP8 stage's cache row, fetched with the other per-request words so that
  // its latency is not paid at the stage's barrier
  int64_t cache_loc = kNoRow;
  if constexpr (kFp8) {
    if (in_batch && (kWarpRows || t == 0)) cache_loc = a.cache_loc[b];
  }
  const int col = 4 * t;
  const InT* in = static_cast<const InT*>(a.input) + static_cast<int64_t>(in_batch ? b : 0) * 2 * D;
  float4 kin[G], sin_[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    kin[g] = In4<InT>::load(in, col + kSpan * g);
    sin_[g] = In4<InT>::load(in + D, col + kSpan * g);
  }
  bool ok = in_batch;
  if (ok && seq_len < 1) {
    if (t == 0) flag_error(a.err, CKV_DEVERR_SEQ_LEN);
    ok = false;
  }
  if (ok && (index < 0 || index >= a.num_slots)) {
    if (t == 0) flag_error(a.err, CKV_DEVERR_SLOT);
    ok = false;
  }
  const int p = ok ? (seq_len - 1) & 127 : 0;  // chunk position of the new token
  float* st = a.state + static_cast<int64_t>(ok ? index : 0) * 3 * D + col;

  float4 ap[G], om[G], os[G], okv[G];
#pragma unroll
  for (int g = 0; g < G; ++g) ap[g] = ld_shared_ro_f4(a.ape + p * D + col + kSpan * g);
  if (ok && p != 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      om[g] = *reinterpret_cast<const float4*>(st + kSpan * g);
      os[g] = *reinterpret_cast<const float4*>(st + D + kSpan * g);
      okv[g] = *reinterpret_cast<const float4*>(st + 2 * D + kSpan * g);
    }
  }
  float4 nm[G], ns[G], nkv[G];
  bool max_same[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    max_same[g] = ok && p != 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float z = get(sin_[g], i) + get(ap[g], i);
      const float k = get(kin[g], i);
      if (p == 0) {
        set(nm[g], i, z);
        set(ns[g], i, 1.f);
        set(nkv[g], i, k);
      } else {
        const float m1 = get(om[g], i);
        const float M = fmaxf(m1, z);
        const float w1 = get(os[g], i) * exp_diff(m1, M);
        const float w2 = exp_diff(z, M);
        const float s = w1 + w2;
        set(nm[g], i, M);
        set(ns[g], i, s);
        set(nkv[g], i, (get(okv[g], i) * w1 + k * w2) / s);
        max_same[g] = max_same[g] && __float_as_uint(M) == __float_as_uint(m1);
      }
    }
    // the 32-byte sector of the max row shared with the partner lane is left
    // as it is (the new bits equal the stored ones) when neither half changed
    max_same[g] = __shfl_xor_sync(0xFFFFFFFFu, max_same[g], 1) && max_same[g];
  }
  // plain stores first, so that their registers are free for the FP8 stage
  constexpr int kBlocks = D / 128;
  if (ok) {
    if (p == 127) {
      if (a.out) {
        float* o = a.out + static_cast<int64_t>(b) * D + col;
#pragma unroll
        for (int g = 0; g < G; ++g) *reinterpret_cast<float4*>(o + kSpan * g) = nkv[g];
      }
    } else {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        if (!max_same[g]) *reinterpret_cast<float4*>(st + kSpan * g) = nm[g];
        *reinterpret_cast<float4*>(st + D + kSpan * g) = ns[g];
        *reinterpret_cast<float4*>(st + 2 * D + kSpan * g) = nkv[g];
      }
    }
  }
  if constexpr (kFp8 && kWarpRows) {
    // the request's warps hold whole blocks in the rotation's lane layout:
    // channels 4l..4l+3 of block t / 32 + (D / 256) g in lane l's group g
    if (ok && p == 127) {  // the same for every thread of the request
      if (cache_loc < 0 || cache_loc >= a.num_pages * a.page_size) {
        if (t == 0) flag_error(a.err, CKV_DEVERR_CACHE_LOC);
      } else {
#pragma unroll
        for (int g = 0; g < G; ++g)
          fp8_block_store(nkv[g], a.cache, a.page_size, cache_loc, kBlocks, t / 32 + (kSpan / 128) * g, t & 31,
                          a.round_scale != 0);
      }
    }
  } else if constexpr (kFp8) {
    // closing rows staged per CTA, then one warp per 128-channel block
    __shared__ __align__(16) float s_row[kRpc][D];
    __shared__ int64_t s_loc[kRpc];
    const int r = threadIdx.x / kTpr;
    const bool closing = ok && p == 127;
    if (closing) {
#pragma unroll
      for (int g = 0; g < G; ++g) *reinterpret_cast<float4*>(&s_row[r][col + kSpan * g]) = nkv[g];
    }
    if (t == 0) s_loc[r] = closing ? cache_loc : kNoRow;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t rows = a.num_pages * a.page_size;
    for (int blk = warp; blk < kRpc * kBlocks; blk += kDecodeThreads / 32) {
      const int rr = blk / kBlocks, j = blk % kBlocks;
      const int64_t loc = s_loc[rr];
      if (loc == kNoRow) continue;
      if (loc < 0 || loc >= rows) {
        if (lane == 0 && j == 0) flag_error(a.err, CKV_DEVERR_CACHE_LOC);
        continue;
      }
      fp8_block_store(&s_row[rr][128 * j], a.cache, a.page_size, loc, kBlocks, j, lane, a.round_scale != 0);
    }
  }
}

// --------------------------------------------------------------------------
// prefill
// --------------------------------------------------------------------------
constexpr int kPrefillWarps = 8;                 // warps per CTA
constexpr int kPosPerWarp = 128 / kPrefillWarps; // chunk positions per warp
constexpr int kBatch = 8;                        // tokens loaded per round

template <int D, typename InT, bool kWrite, bool kFp8>
__global__ void __launch_bounds__(kPrefillWarps * 32, 2)
    c128_prefill_kernel(const __grid_constant__ C128PrefillArgs a) {
  static_assert(!(kWrite && kFp8), "the FP8 output stage belongs to the compress pass");
  static_assert(kPrefillWarps * 32 >= 128, "the epilogue's 128 threads own one channel of the slice each");
  constexpr int S = D / 128;  // 128-channel slices per row
  __shared__ __align__(16) float4 s_m[kPrefillWarps][32];
  __shared__ __align__(16) float4 s_s[kPrefillWarps][32];
  __shared__ __align__(16) float4 s_a[kPrefillWarps][32];

  // The write pass chained to this call's compress pass reads its plan,
  // indices and tokens before the dependency wait (none of them is written by
  // the compress pass, and everything before that pass was complete when it
  // let this grid launch), so its token reduction overlaps the compress pass;
  // it waits only before the state.  Otherwise: wait first.
  const bool early = kWrite && a.write_early;
  if (!early) pdl_wait();
  const uint32_t plan_id = blockIdx.x / S;
  const int slice = blockIdx.x % S;
  const uint32_t n_host = kWrite ? a.num_write : a.num_compress;
  const uint32_t n_plans = a.counts ? min(a.counts[kWrite ? 1 : 0], n_host) : n_host;
  if (plan_id >= n_plans) return;
  const uint4 raw = *reinterpret_cast<const uint4*>(kWrite ? a.write_plan + plan_id
                                                           : a.compress_plan + plan_id);
  pdl_trigger();
  const uint32_t ragged_id = raw.x, batch = raw.y, position = raw.z, window = raw.w;
  if (ragged_id == 0xFFFFFFFFu) return;  // sentinel (graph padding)

  const uint32_t pic = position & 127u;  // chunk position of the last token
  const bool plan_ok = batch < static_cast<uint32_t>(a.B) && window >= 1 && window <= pic + 1 &&
                       ragged_id < a.num_tokens && ragged_id + 1 >= window &&
                       (kWrite ? (pic != 127u) : (pic == 127u));
  if (!plan_ok) {
    if (threadIdx.x == 0) flag_error(a.err, CKV_DEVERR_PLAN);
    return;
  }
  const int chunk_offset = static_cast<int>(pic + 1 - window);
  const int window_end = static_cast<int>(pic + 1);
  // the FP8 stage's cache row, fetched now so that the CTA does not end on its latency
  int64_t fp8_loc = 0;
  if constexpr (kFp8) {
    if (threadIdx.x < 32) fp8_loc = a.cache_loc[ragged_id];
  }
  int32_t load_index = -1, store_index = -1;
  if (chunk_offset != 0) load_index = a.load_indices[batch];
  if (kWrite) store_index = a.indices[batch];
  if ((chunk_offset != 0 && (load_index < 0 || load_index >= a.num_slots)) ||
      (kWrite && (store_index < 0 || store_index >= a.num_slots))) {
    if (threadIdx.x == 0) flag_error(a.err, CKV_DEVERR_SLOT);
    return;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int col = slice * 128 + 4 * lane;
  const int64_t row_c0 = static_cast<int64_t>(ragged_id) - pic;  // ragged row of chunk position 0
  const InT* in = static_cast<const InT*>(a.input);

  float M[4] = {kNegBig, kNegBig, kNegBig, kNegBig};
  float Ssum[4] = {0.f, 0.f, 0.f, 0.f}, A[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int r = 0; r < kPosPerWarp / kBatch; ++r) {
    const int j0 = warp * kPosPerWarp + r * kBatch;
    if (j0 >= window_end || j0 + kBatch <= chunk_offset) continue;  // warp-uniform
    float4 kv[kBatch], sc[kBatch], ap[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int j = j0 + i;
      if (j >= chunk_offset && j < window_end) {
        const InT* row = in + (row_c0 + j) * 2 * D;
        kv[i] = In4<InT>::load(row, col);
        sc[i] = In4<InT>::load(row + D, col);
        ap[i] = ld_shared_ro_f4(a.ape + j * D + col);
      } else {
        kv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        sc[i] = make_float4(kNegBig, kNegBig, kNegBig, kNegBig);
        ap[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float z[kBatch];
      float bm = kNegBig;
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        z[i] = get(sc[i], c) + get(ap[i], c);
        bm = fmaxf(bm, z[i]);
      }
      float bs = 0.f, ba = 0.f;
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int j = j0 + i;
        const float e = (j >= chunk_offset && j < window_end) ? exp_diff(z[i], bm) : 0.f;
        bs += e;
        ba = fmaf(e, get(kv[i], c), ba);
      }
      const float nm = fmaxf(M[c], bm);
      const float f1 = exp_diff(M[c], nm), f2 = exp_diff(bm, nm);
      Ssum[c] = Ssum[c] * f1 + bs * f2;
      A[c] = A[c] * f1 + ba * f2;
      M[c] = nm;
    }
  }
  s_m[warp][lane] = make_float4(M[0], M[1], M[2], M[3]);
  s_s[warp][lane] = make_float4(Ssum[0], Ssum[1], Ssum[2], Ssum[3]);
  s_a[warp][lane] = make_float4(A[0], A[1], A[2], A[3]);
  __syncthreads();
  if (threadIdx.x >= 128) return;

  // Channel t of the slice: merge the 8 warp partials, then the stored partial.
  const int t = threadIdx.x;
  const float* fm = reinterpret_cast<const float*>(s_m);
  const float* fs = reinterpret_cast<const float*>(s_s);
  const float* fa = reinterpret_cast<const float*>(s_a);
  float m = kNegBig;
#pragma unroll
  for (int w = 0; w < kPrefillWarps; ++w) m = fmaxf(m, fm[w * 128 + t]);
  float ssum = 0.f, acc = 0.f;
#pragma unroll
  for (int w = 0; w < kPrefillWarps; ++w) {
    const float f = exp_diff(fm[w * 128 + t], m);
    ssum = fmaf(fs[w * 128 + t], f, ssum);
    acc = fmaf(fa[w * 128 + t], f, acc);
  }
  float kv = acc / ssum;
  const int ch = slice * 128 + t;
  if (early) pdl_wait();
  if (chunk_offset != 0) {
    const float* ld = a.state + static_cast<int64_t>(load_index) * 3 * D + ch;
    const float m1 = ld[0], s1 = ld[D], k1 = ld[2 * D];
    const float nm = fmaxf(m1, m);
    const float w1 = s1 * exp_diff(m1, nm), w2 = ssum * exp_diff(m, nm);
    ssum = w1 + w2;
    kv = (k1 * w1 + kv * w2) / ssum;
    m = nm;
  }
  if (kWrite) {
    float* stp = a.state + static_cast<int64_t>(store_index) * 3 * D + ch;
    stp[0] = m;
    stp[D] = ssum;
    stp[2 * D] = kv;
  } else {
    if (a.out) a.out[static_cast<int64_t>(ragged_id) * D + ch] = kv;
    if constexpr (kFp8) {
      // the slice is block `slice` of the row: staged, then warp 0 stores it
      __shared__ __align__(16) float s_row[128];
      s_row[t] = kv;
      asm volatile("bar.sync 1, 128;" ::: "memory");  // the 128 epilogue threads
      if (t < 32) {
        const int64_t loc = fp8_loc;
        if (loc < 0 || loc >= a.num_pages * a.page_size) {
          if (t == 0 && slice == 0) flag_error(a.err, CKV_DEVERR_CACHE_LOC);
        } else {
          fp8_block_store(s_row, a.cache, a.page_size, loc, S, slice, t, a.round_scale != 0);
        }
      }
    }
  }
}

template <int D, typename InT>
cudaError_t decode_d(const C128DecodeArgs& a, bool use_pdl, cudaStream_t s) {
  constexpr int G = kDecodeGroups, kRpc = kDecodeThreads / (D / (4 * G));
  const dim3 grid((a.B + kRpc - 1) / kRpc);
  if (a.cache)
    return launch_ex(c128_decode_kernel<D, InT, G, kDecodeFp8MinBlocks, true>, grid, dim3(kDecodeThreads), 0,
                     use_pdl, s, a);
  return launch_ex(c128_decode_kernel<D, InT, G, kDecodeMinBlocks, false>, grid, dim3(kDecodeThreads), 0, use_pdl, s,
                   a);
}

// Automatic choice: the persistent TMA pipeline from 1024 compress segments
// (measured, one request from position 0: the one-CTA-per-segment kernel is
// faster up to 512 segments -- its CTAs need no bias staging or pipeline fill
// -- the two are equal for fp32 at 2048 and the pipeline is 7% faster for
// bf16 at 2048 and 13% at 8192).
constexpr uint32_t kTmaMinSegments = 1024;

template <int D, typename InT>
cudaError_t prefill_d(const C128PrefillArgs& a, bool use_pdl, cudaStream_t s) {
  constexpr int S = D / 128;
  constexpr int dtype = std::is_same<InT, float>::value ? CKV_F32 : CKV_BF16;
  if (a.num_compress) {
    const int v = prefill_variant();
    cudaError_t e = cudaErrorNotSupported;
    const bool tma = v == 2 || (v == 0 && a.num_compress >= kTmaMinSegments);
    if (tma && c128_prefill_tma_supported(a, D, dtype)) {
      e = launch_c128_prefill_compress_tma(a, D, dtype, use_pdl, s);
      if (e == cudaErrorNotSupported) (void)cudaGetLastError();
    }
    if (e == cudaErrorNotSupported) {
      const dim3 grid(static_cast<unsigned>(a.num_compress) * S);
      e = a.cache ? launch_ex(c128_prefill_kernel<D, InT, false, true>, grid, dim3(kPrefillWarps * 32), 0, use_pdl, s,
                              a)
                  : launch_ex(c128_prefill_kernel<D, InT, false, false>, grid, dim3(kPrefillWarps * 32), 0, use_pdl,
                              s, a);
    }
    if (e != cudaSuccess) return e;
  }
  if (a.num_write) {
    const dim3 grid(static_cast<unsigned>(a.num_write) * S);
    C128PrefillArgs w = a;
    w.write_early = (use_pdl && a.num_compress) ? 1 : 0;
    cudaError_t e =
        launch_ex(c128_prefill_kernel<D, InT, true, false>, grid, dim3(kPrefillWarps * 32), 0, use_pdl, s, w);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_c128_decode(const C128DecodeArgs& a, int D, int in_dtype, bool use_pdl,
                               cudaStream_t s) {
  if (in_dtype == CKV_F32) {
    if (D == 128) return decode_d<128, float>(a, use_pdl, s);
    if (D == 256) return decode_d<256, float>(a, use_pdl, s);
    if (D == 512) return decode_d<512, float>(a, use_pdl, s);
  } else {
    if (D == 128) return decode_d<128, __nv_bfloat16>(a, use_pdl, s);
    if (D == 256) return decode_d<256, __nv_bfloat16>(a, use_pdl, s);
    if (D == 512) return decode_d<512, __nv_bfloat16>(a, use_pdl, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_c128_prefill(const C128PrefillArgs& a, int D, int in_dtype, bool use_pdl,
                                cudaStream_t s) {
  if (in_dtype == CKV_F32) {
    if (D == 128) return prefill_d<128, float>(a, use_pdl, s);
    if (D == 256) return prefill_d<256, float>(a, use_pdl, s);
    if (D == 512) return prefill_d<512, float>(a, use_pdl, s);
  } else {
    if (D == 128) return prefill_d<128, __nv_bfloat16>(a, use_pdl, s);
    if (D == 256) return prefill_d<256, __nv_bfloat16>(a, use_pdl, s);
    if (D == 512) return prefill_d<512, __nv_bfloat16>(a, use_pdl, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace ckv
