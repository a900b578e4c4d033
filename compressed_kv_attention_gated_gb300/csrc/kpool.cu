// kpool.cu -- pooled (P <= 16, D = 128) gated-softmax compression kernels.
//
// Source: vLLM page "vllm.models.glm5next.amd.ops.kpool_compress"
// (_kpool_decode_update_batched_kernel, _kpool_softmax_rotate_write_cache_kernel,
// _kpool_tail_seed_kernel).  Those are AMD Triton kernels with one program per
// request/pool and a 128-wide block; the design here is our own for sm_103a:
//
//   * one-shot: one warp per pool, lane l owning channels 4l..4l+3, so every
//     key/score slot row (256 B of bf16) is one coalesced 8-byte-per-lane load
//     and every FP8 output row (128 B) one 4-byte-per-lane store; all P slot
//     rows of a pool are loaded before any arithmetic (P * 16 B in flight per
//     lane), the per-slot bias table is staged in shared memory once per CTA;
//   * decode: one CTA of two warps per request, thread t owning the channel
//     pair (2t, 2t + 1) (described at the kernel);
//   * exact two-pass softmax from registers: z = score + ape for the P slots,
//     max, then one ex2 per element;
//   * for large batches, a persistent variant in which every warp streams its
//     pools through a private three-stage ring of shared-memory buffers with 1-D
//     bulk copies (cp.async.bulk, completion on an mbarrier), so the next
//     pool's 8 KB arrive while the current one is reduced, rotated and packed;
//   * Hadamard-128: two butterfly spans inside the lane (1, 2), then five
//     warp-shuffle spans (4..64 = lane masks 1..16), ascending; the absmax as
//     one warp max-reduction of the values' bit patterns; fused FP8-e4m3
//     packing (cvt.rn.satfinite) and cache write.
//
// The pooled path is memory bound (no dense contraction); no tensor cores.
#include "ckv_device.cuh"
#include "ckv_fp8.cuh"
#include "ckv_launch.h"
#include "ckv_launch_util.cuh"
#include "ckv_tma.cuh"

namespace ckv {
namespace {

constexpr int kD = 128;          // pooled head dim (the rotation is 128-point)
constexpr int kRowBytes = kD + 4; // FP8 row + fp32 scale per cache row

// Pairs of fp32 in one 64-bit register pair, for sm_100+'s packed fp32 ops:
// each packed op is two independent IEEE round-to-nearest operations, so it
// gives bit for bit what two scalar ones give, in one instruction.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// two bf16 (low half first) widened to a packed fp32 pair
__device__ __forceinline__ uint64_t f2_from_bf16x2(uint32_t w) { return f2_pack(bf16_lo(w), bf16_hi(w)); }

// Softmax-weighted pool of P slots for the lane's 4 channels.
// kr/sr: slot rows of keys/scores, 4 bf16 each; s_ape2: [P][128] fp32 in smem,
// the bias already multiplied by log2(e), so each logit in the log2 domain is
// one FMA (score * log2(e) + bias') and each weight one ex2 of a difference.
// Channels (0, 1) and (2, 3) of the lane travel as packed pairs through the
// FMAs and additions; max and ex2 are scalar.
template <int P>
__device__ __forceinline__ void pool_softmax(const uint2 (&kr)[P], const uint2 (&sr)[P],
                                             const float* s_ape2, int lane, float (&x)[4]) {
  const uint64_t log2e2 = f2_pack(kLog2e, kLog2e);
  uint64_t z[P][2];
  float m[4] = {kNegBig, kNegBig, kNegBig, kNegBig};
#pragma unroll
  for (int j = 0; j < P; ++j) {
    const float4 a = reinterpret_cast<const float4*>(s_ape2 + j * kD)[lane];
    z[j][0] = f2_fma(f2_from_bf16x2(sr[j].x), log2e2, f2_pack(a.x, a.y));
    z[j][1] = f2_fma(f2_from_bf16x2(sr[j].y), log2e2, f2_pack(a.z, a.w));
    float z0, z1, z2, z3;
    f2_unpack(z[j][0], z0, z1);
    f2_unpack(z[j][1], z2, z3);
    m[0] = fmaxf(m[0], z0);
    m[1] = fmaxf(m[1], z1);
    m[2] = fmaxf(m[2], z2);
    m[3] = fmaxf(m[3], z3);
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint64_t mh = f2_pack(m[2 * h], m[2 * h + 1]);
    uint64_t den = f2_pack(0.f, 0.f), acc = den;
#pragma unroll
    for (int j = 0; j < P; ++j) {
      float t0, t1;
      f2_unpack(f2_sub(z[j][h], mh), t0, t1);
      const uint64_t e = f2_pack(fast_exp2(t0), fast_exp2(t1));
      den = f2_add(den, e);
      acc = f2_fma(e, f2_from_bf16x2(h ? kr[j].y : kr[j].x), acc);
    }
    float d0, d1, a0, a1;
    f2_unpack(den, d0, d1);
    f2_unpack(acc, a0, a1);
    x[2 * h] = __fdividef(a0, d0);  // den in [1, P]
    x[2 * h + 1] = __fdividef(a1, d1);
  }
}

__device__ __forceinline__ void write_taps(float* tx, uint16_t* txb, uint16_t* tyb, int64_t row,
                                           int lane, const float (&x)[4], const float (&xb)[4],
                                           const float (&yb)[4]) {
  if (tx) reinterpret_cast<float4*>(tx + row * kD)[lane] = make_float4(x[0], x[1], x[2], x[3]);
  if (txb)
    reinterpret_cast<uint2*>(txb + row * kD)[lane] =
        make_uint2(pack_bf16x2_rn(xb[0], xb[1]), pack_bf16x2_rn(xb[2], xb[3]));
  if (tyb)
    reinterpret_cast<uint2*>(tyb + row * kD)[lane] =
        make_uint2(pack_bf16x2_rn(yb[0], yb[1]), pack_bf16x2_rn(yb[2], yb[3]));
}

// Where cache row loc lives: its kD code bytes and its fp32 scale.  Computed
// as soon as loc is known, so that the 64-bit division is off the path
// between a pool's arithmetic and its store.
struct CacheRow {
  uint8_t* codes;
  float* scale;
};

// page = loc / page_size, by a shift when page_size is a power of two
// (page_shift >= 0): a 64-bit division is a long instruction sequence
__device__ __forceinline__ int64_t page_of(int64_t loc, int64_t page_size, int32_t page_shift) {
  return page_shift >= 0 ? (loc >> page_shift) : loc / page_size;
}

__device__ __forceinline__ CacheRow cache_row(uint8_t* cache, int64_t page_size, int32_t page_shift, int64_t loc) {
  const int64_t page = page_of(loc, page_size, page_shift), tok = loc - page * page_size;
  uint8_t* base = cache + page * page_size * kRowBytes;
  return {base + tok * kD, reinterpret_cast<float*>(base + page_size * kD) + tok};
}

__device__ __forceinline__ void cache_write(const CacheRow& row, int lane, uint32_t codes, float scale) {
  reinterpret_cast<uint32_t*>(row.codes)[lane] = codes;
  if (lane == 0) *row.scale = scale;
}

// The same with the address formed at the store (the bulk pipeline: holding
// the address across its wait costs registers and measured slower).
__device__ __forceinline__ void cache_write(uint8_t* cache, int64_t page_size, int32_t page_shift, int64_t loc,
                                            int lane, uint32_t codes, float scale) {
  const int64_t page = page_of(loc, page_size, page_shift), tok = loc - page * page_size;
  uint8_t* base = cache + page * page_size * kRowBytes;
  reinterpret_cast<uint32_t*>(base + tok * kD)[lane] = codes;
  if (lane == 0) *reinterpret_cast<float*>(base + page_size * kD + 4 * tok) = scale;
}

// Stage the [P][128] bias table in shared memory, multiplied by log2(e), and
// let the next grid in the stream begin launching.  The caller has waited for
// the preceding grid (programmatic dependent launch; a no-op otherwise) and
// has usually issued its first row loads already, so that their latency and
// the staging overlap.
template <int P>
__device__ __forceinline__ void stage_ape(float* s_ape2, const float* ape) {
  for (int i = threadIdx.x; i < P * kD / 4; i += blockDim.x) {
    float4 v = ld_shared_ro_f4(ape + 4 * i);
    v.x *= kLog2e;
    v.y *= kLog2e;
    v.z *= kLog2e;
    v.w *= kLog2e;
    reinterpret_cast<float4*>(s_ape2)[i] = v;
  }
  __syncthreads();
  pdl_trigger();
}

constexpr int kWarpsPerCta = 8;

// One-shot pooled compression: warp w of CTA c handles pool c*8 + w.
template <int P, bool kRound>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
    kpool_compress_kernel(const __grid_constant__ KpoolCompressArgs a) {
  __shared__ __align__(16) float s_ape[P * kD];
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t pool = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5);
  const bool want = pool < a.n_pools && (!a.write_mask || a.write_mask[pool] != 0);
  // the rows and the cache location are in flight while the bias is staged
  int64_t loc = 0;
  uint2 kr[P], sr[P];
  if (want) {
    loc = a.write_cache ? a.loc[pool] : 0;
    const uint16_t* kb = a.slot_k + pool * P * kD + 4 * lane;
    const uint16_t* sb = a.slot_score + pool * P * kD + 4 * lane;
#pragma unroll
    for (int j = 0; j < P; ++j) {
      kr[j] = ld_stream_u2(kb + j * kD);
      sr[j] = ld_stream_u2(sb + j * kD);
    }
  }
  stage_ape<P>(s_ape, a.ape);
  if (!want) return;
  const bool loc_ok = a.write_cache && loc >= 0 && loc < a.num_pages * a.page_size;
  const CacheRow row = loc_ok ? cache_row(a.cache, a.page_size, a.page_shift, loc) : CacheRow{nullptr, nullptr};
  float x[4], xb[4], yb[4], scale;
  uint32_t codes;
  pool_softmax<P>(kr, sr, s_ape, lane, x);
  rotate_quantize<kRound>(x, lane, codes, scale, xb, yb);

  if (a.write_cache) {
    if (!loc_ok) {
      if (lane == 0) flag_error(a.err, CKV_DEVERR_CACHE_LOC);
    } else {
      cache_write(row, lane, codes, scale);
    }
  }
  if (a.out_fp8) {
    reinterpret_cast<uint32_t*>(a.out_fp8 + pool * kD)[lane] = codes;
    if (lane == 0) a.out_scale[pool] = scale;
  }
  write_taps(a.tap_x, a.tap_xb, a.tap_yb, pool, lane, x, xb, yb);
}

// One-shot pooled compression, persistent and bulk-copy fed.  Warp g (of W in
// the grid) handles pools g, g + W, g + 2W, ...; each pool's P key rows and P
// score rows (contiguous, P * 256 B each) are copied into one of the warp's
// kBulkStages shared-memory stages by lane 0 (up to kBulkStages - 1 pools
// ahead of the one being reduced), and the whole warp waits on the stage's
// mbarrier before reading it.  Pools masked out by write_mask are
// neither copied nor computed.  Waits are bounded; a timeout flags
// CKV_DEVERR_TIMEOUT, drains the warp's own copies and leaves.
template <int P, int kBulkWarps, int kBulkStages>
struct BulkLayout {
  static constexpr int kPoolBytes = P * kD * 2;  // one array of one pool
  static constexpr int kApe = 0;
  static constexpr int kBuf = P * kD * 4;
  static constexpr int kBar = kBuf + kBulkWarps * kBulkStages * 2 * kPoolBytes;
  static constexpr int kBytes = kBar + kBulkWarps * kBulkStages * 8;
};

template <int P, bool kRound, int kBulkWarps, int kBulkStages>
__global__ void __launch_bounds__(kBulkWarps * 32, 1)
    kpool_compress_bulk_kernel(const __grid_constant__ KpoolCompressArgs a) {
  using L = BulkLayout<P, kBulkWarps, kBulkStages>;
  extern __shared__ __align__(128) uint8_t smem[];
  float* s_ape = reinterpret_cast<float*>(smem + L::kApe);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* mybuf = smem + L::kBuf + warp * kBulkStages * 2 * L::kPoolBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar) + warp * kBulkStages;
  if (lane == 0) {
    for (int s = 0; s < kBulkStages; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  pdl_wait();

  const int64_t W = static_cast<int64_t>(gridDim.x) * kBulkWarps;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kBulkWarps + warp;
  auto wanted = [&](int64_t pool) { return pool < a.n_pools && (!a.write_mask || a.write_mask[pool] != 0); };
  auto issue = [&](int64_t pool, int s) {
    uint8_t* dst = mybuf + s * 2 * L::kPoolBytes;
    mbar_arrive_expect_tx(&bars[s], 2 * L::kPoolBytes);
    bulk_load(dst, a.slot_k + pool * P * kD, L::kPoolBytes, &bars[s]);
    bulk_load(dst + L::kPoolBytes, a.slot_score + pool * P * kD, L::kPoolBytes, &bars[s]);
  };
  uint32_t parity = 0, armed = 0;  // per-stage bits
  if (lane == 0) {
    for (int s = 0; s < kBulkStages; ++s) {
      const int64_t pool = first + s * W;
      if (wanted(pool)) issue(pool, s);
    }
  }
  for (int s = 0; s < kBulkStages; ++s)
    if (wanted(first + s * W)) armed |= 1u << s;
  stage_ape<P>(s_ape, a.ape);  // overlaps the first copies; ends with __syncthreads()

  // cache locations are fetched one pool ahead so that no global load sits
  // between a pool's arithmetic and its store
  int64_t loc_next = (a.write_cache && first < a.n_pools) ? a.loc[first] : 0;
  int s = 0;
  for (int64_t pool = first; pool < a.n_pools; pool += W) {
    const int64_t loc = loc_next;
    if (a.write_cache && pool + W < a.n_pools) loc_next = a.loc[pool + W];
    if (armed & (1u << s)) {
      if (!mbar_wait(&bars[s], (parity >> s) & 1u)) {
        if (lane == 0) flag_error(a.err, CKV_DEVERR_TIMEOUT);
        for (int x = 0; x < kBulkStages; ++x)
          if (x != s && (armed & (1u << x))) (void)mbar_wait(&bars[x], (parity >> x) & 1u);
        return;
      }
      parity ^= 1u << s;
      armed &= ~(1u << s);
      const uint8_t* kb = mybuf + s * 2 * L::kPoolBytes;
      const uint8_t* sb = kb + L::kPoolBytes;
      uint2 kr[P], sr[P];
#pragma unroll
      for (int j = 0; j < P; ++j) {
        kr[j] = reinterpret_cast<const uint2*>(kb + j * kD * 2)[lane];
        sr[j] = reinterpret_cast<const uint2*>(sb + j * kD * 2)[lane];
      }
      __syncwarp();
      // the stage is free again: prefetch the pool kBulkStages turns ahead
      const int64_t ahead = pool + kBulkStages * W;
      if (wanted(ahead)) {
        if (lane == 0) {
          fence_proxy_async_smem();
          issue(ahead, s);
        }
        armed |= 1u << s;
      }
      float x[4], xb[4], yb[4], scale;
      uint32_t codes;
      pool_softmax<P>(kr, sr, s_ape, lane, x);
      rotate_quantize<kRound>(x, lane, codes, scale, xb, yb);
      if (a.write_cache) {
        if (loc < 0 || loc >= a.num_pages * a.page_size) {
          if (lane == 0) flag_error(a.err, CKV_DEVERR_CACHE_LOC);
        } else {
          cache_write(a.cache, a.page_size, a.page_shift, loc, lane, codes, scale);
        }
      }
      if (a.out_fp8) {
        reinterpret_cast<uint32_t*>(a.out_fp8 + pool * kD)[lane] = codes;
        if (lane == 0) a.out_scale[pool] = scale;
      }
      write_taps(a.tap_x, a.tap_xb, a.tap_yb, pool, lane, x, xb, yb);
    } else {
      const int64_t ahead = pool + kBulkStages * W;
      if (wanted(ahead)) {
        if (lane == 0) issue(ahead, s);
        armed |= 1u << s;
      }
    }
    if (++s == kBulkStages) s = 0;
  }
}

// Decode / verify update: one CTA of two warps per request, thread t owning
// channels 2t and 2t + 1 of the pooled key (one bf16 pair: every row access
// is a 4-byte access per thread, 256 B per CTA).  The request's tokens are
// walked in order, kPrefetch at a time; all 64 threads load the group's index
// words (the same words: broadcast) and their pair of the group's key and
// score rows.  A closing pool's ring rows and bias are loaded together (the
// one round trip that depends on the index words) and its cache row is
// located while they are in flight; its arithmetic is
// deferred until the stashes of the later tokens of the group (or, after the
// last group, of the request) have been issued, so those stores are not left
// at the end of the critical path.  A thread's later store to a ring slot
// cannot overtake its own earlier load of it (same thread, same address), and
// the pool takes its current token from registers, so deferring is safe.  The
// arithmetic per channel is that of the one-shot kernels (same operations,
// same order), so both give identical rows.  A request's branch decisions
// come from words both warps read alike, so the barrier inside a pool's
// rotation is reached by the whole CTA.
constexpr int kPrefetch = 4;
constexpr int kDecThreads = kD / 2;  // two channels per thread

// bf16 -> Hadamard-128 -> bf16 -> absmax FP8 of a 128-channel vector held as
// channel pairs (2t, 2t + 1) by the 64 threads of a CTA.  Butterfly spans 1
// (inside the thread), 2..32 (lane shuffles), 64 (the other warp, through
// shared memory), each (u + v, u - v) in fp32, then one multiply by
// fp32(1/sqrt(128)): the rotation of rotate_quantize, element for element.
// After the one exchange each thread also forms the last stage of its
// partner's pair, so every warp holds all 128 outputs (4 per lane) and the
// absmax is one warp reduction, with no second exchange.  Every thread of the
// CTA must call it.
template <bool kRound>
__device__ __forceinline__ void rotate_quantize_pair(float x0, float x1, int t, float2* s_x, uint32_t& codes,
                                                     float& scale, float (&xb)[2], float (&yb)[2]) {
  const int lane = t & 31;
  xb[0] = round_bf16(x0);
  xb[1] = round_bf16(x1);
  float a0 = xb[0] + xb[1];  // span 1
  float a1 = xb[0] - xb[1];
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {  // spans 2..32: partner lane l ^ m
    // lower channel: a + o; upper channel: o - a, rounded once like a subtraction
    const float o0 = __shfl_xor_sync(0xFFFFFFFFu, a0, m);
    const float o1 = __shfl_xor_sync(0xFFFFFFFFu, a1, m);
    const float sgn = (lane & m) ? -1.f : 1.f;
    a0 = fmaf(a0, sgn, o0);
    a1 = fmaf(a1, sgn, o1);
  }
  s_x[t] = make_float2(a0, a1);  // span 64: the pair of thread t ^ 32
  __syncthreads();
  const float2 p = s_x[t ^ 32];
  float f0, f1, g0, g1;  // this thread's outputs, and its partner's
  if (t < 32) {
    f0 = a0 + p.x, f1 = a1 + p.y, g0 = a0 - p.x, g1 = a1 - p.y;
  } else {
    f0 = p.x - a0, f1 = p.y - a1, g0 = p.x + a0, g1 = p.y + a1;
  }
  const float c = __uint_as_float(0x3DB504F3u);  // fp32(1/sqrt(128))
  yb[0] = round_bf16(f0 * c);
  yb[1] = round_bf16(f1 * c);
  float am = fmaxf(fmaxf(fabsf(yb[0]), fabsf(yb[1])), fmaxf(fabsf(round_bf16(g0 * c)), fabsf(round_bf16(g1 * c))));
  am = fmaxf(warp_absmax(am), 1e-4f);
  const float v = am * __uint_as_float(0x3B124925u);  // absmax * fp32(1/448)
  float q0, q1;
  if (kRound) {
    // smallest power of two >= v; its exact reciprocal gives the IEEE quotient
    const uint32_t bits = __float_as_uint(v);
    const uint32_t e = (bits & 0x007FFFFFu) ? (bits & 0x7F800000u) + 0x00800000u : (bits & 0x7F800000u);
    scale = __uint_as_float(e);
    const float inv = __uint_as_float((254u << 23) - e);
    q0 = fminf(fmaxf(yb[0] * inv, -448.f), 448.f);
    q1 = fminf(fmaxf(yb[1] * inv, -448.f), 448.f);
  } else {
    scale = v;
    q0 = fminf(fmaxf(__fdiv_rn(yb[0], scale), -448.f), 448.f);
    q1 = fminf(fmaxf(__fdiv_rn(yb[1], scale), -448.f), 448.f);
  }
  codes = __nv_cvt_float2_to_fp8x2(make_float2(q0, q1), __NV_SATFINITE, __NV_E4M3) & 0xFFFFu;
}

template <int P, bool kRound>
__global__ void __launch_bounds__(kDecThreads)
    kpool_decode_kernel(const __grid_constant__ KpoolDecodeArgs a) {
  __shared__ float2 s_x[kDecThreads];
  pdl_wait();
  const int t = threadIdx.x;
  const int b = blockIdx.x;
  const int64_t cache_rows = a.num_pages * a.page_size;
  const uint16_t* key = a.key + b * a.key_sb + 2 * t;
  const uint16_t* score = a.score + b * a.score_sb + 2 * t;

  int32_t loc[kPrefetch], pos[kPrefetch], tslot[kPrefetch];
  uint32_t kc[kPrefetch], sc[kPrefetch];  // bf16 pairs of this thread's channels
  auto load_group = [&](int t0) {
#pragma unroll
    for (int i = 0; i < kPrefetch; ++i) {
      const int tk = t0 + i;
      if (tk < a.N) {
        const int64_t idx = static_cast<int64_t>(b) * a.N + tk;
        loc[i] = __ldg(a.slot_mapping + idx);
        pos[i] = __ldg(a.positions + idx);
        tslot[i] = __ldg(a.tail_slot_mapping + idx);
        kc[i] = __ldg(reinterpret_cast<const uint32_t*>(key + tk * a.key_st));
        sc[i] = __ldg(reinterpret_cast<const uint32_t*>(score + tk * a.score_st));
      } else {
        loc[i] = pos[i] = tslot[i] = -1;  // past N: neither closes nor stashes
        kc[i] = sc[i] = 0u;
      }
    }
  };
  load_group(0);
  pdl_trigger();

  // the pool waiting for its arithmetic: its rows, bias, cache row and tap row
  bool pend = false;
  int64_t pend_row = 0;
  CacheRow pend_cache{nullptr, nullptr};
  uint32_t kr[P], sr[P];
  float2 ap[P];
  auto finish = [&]() {
    const uint64_t log2e2 = f2_pack(kLog2e, kLog2e);
    uint64_t z[P];
    float m0 = kNegBig, m1 = kNegBig;
#pragma unroll
    for (int j = 0; j < P; ++j) {
      z[j] = f2_fma(f2_from_bf16x2(sr[j]), log2e2, f2_pack(ap[j].x * kLog2e, ap[j].y * kLog2e));
      float z0, z1;
      f2_unpack(z[j], z0, z1);
      m0 = fmaxf(m0, z0);
      m1 = fmaxf(m1, z1);
    }
    const uint64_t mm = f2_pack(m0, m1);
    uint64_t den = f2_pack(0.f, 0.f), acc = den;
#pragma unroll
    for (int j = 0; j < P; ++j) {
      float t0, t1;
      f2_unpack(f2_sub(z[j], mm), t0, t1);
      const uint64_t e = f2_pack(fast_exp2(t0), fast_exp2(t1));
      den = f2_add(den, e);
      acc = f2_fma(e, f2_from_bf16x2(kr[j]), acc);
    }
    float d0, d1, a0, a1;
    f2_unpack(den, d0, d1);
    f2_unpack(acc, a0, a1);
    const float x0 = __fdividef(a0, d0), x1 = __fdividef(a1, d1);  // den in [1, P]
    float xb[2], yb[2], scale;
    uint32_t codes;
    rotate_quantize_pair<kRound>(x0, x1, t, s_x, codes, scale, xb, yb);
    reinterpret_cast<uint16_t*>(pend_cache.codes)[t] = static_cast<uint16_t>(codes);
    if (t == 0) *pend_cache.scale = scale;
    if (a.tap_x) reinterpret_cast<float2*>(a.tap_x + pend_row * kD)[t] = make_float2(x0, x1);
    if (a.tap_xb) reinterpret_cast<uint32_t*>(a.tap_xb + pend_row * kD)[t] = pack_bf16x2_rn(xb[0], xb[1]);
    if (a.tap_yb) reinterpret_cast<uint32_t*>(a.tap_yb + pend_row * kD)[t] = pack_bf16x2_rn(yb[0], yb[1]);
    pend = false;
  };

  for (int t0 = 0; t0 < a.N; t0 += kPrefetch) {
    if (t0 > 0) load_group(t0);
#pragma unroll
    for (int i = 0; i < kPrefetch; ++i) {
      const int slot = max(pos[i], 0) & (P - 1);
      const bool pos_valid = loc[i] >= 0 && pos[i] >= 0;
      const bool stash_valid = pos[i] >= 0 && tslot[i] >= 0;
      const bool closes = pos_valid && slot == P - 1;
      if (!closes && !stash_valid) continue;
      const int64_t block = static_cast<int64_t>(max(tslot[i], 0)) / P;
      if (block >= a.num_blocks) {
        if (t == 0) flag_error(a.err, CKV_DEVERR_TAIL_BLOCK);
        continue;
      }
      uint32_t* kring = reinterpret_cast<uint32_t*>(a.ring + block * 2 * P * kD) + t;
      uint32_t* sring = kring + P * kD / 2;
      if (closes) {
        if (loc[i] >= cache_rows) {
          if (t == 0) flag_error(a.err, CKV_DEVERR_CACHE_LOC);
        } else {
          if (pend) finish();  // an earlier pool of this call (P < N): its registers are needed
#pragma unroll
          for (int j = 0; j < P - 1; ++j) {
            kr[j] = kring[j * (kD / 2)];
            sr[j] = sring[j * (kD / 2)];
          }
          kr[P - 1] = kc[i];
          sr[P - 1] = sc[i];
#pragma unroll
          for (int j = 0; j < P; ++j) ap[j] = __ldg(reinterpret_cast<const float2*>(a.ape + j * kD) + t);
          pend = true;
          // the division overlaps the ring read here; a shift measured slower
          pend_cache = cache_row(a.cache, a.page_size, -1, loc[i]);
          pend_row = static_cast<int64_t>(b) * a.N + t0 + i;
        }
      }
      if (stash_valid) {
        kring[slot * (kD / 2)] = kc[i];
        sring[slot * (kD / 2)] = sc[i];
      }
    }
  }
  if (pend) finish();
}

// Tail-ring seed: each warp takes 128 consecutive prefill tokens, 4 per lane.
// Lane l reads the tail slots of tokens 4l..4l+3 and of the tokens P places
// ahead (one 16-byte load each when P is a multiple of 4 and the slot map is
// 16-byte aligned); the tokens among their request's last P are compacted into
// a per-warp list in shared memory, and the warp then copies the listed key
// and score rows (256 B each, 32 lanes x 8 B) with kSeedBatch independent
// loads per lane in flight before their stores, rather than one row at a time.
constexpr int kSeedTokensPerWarp = 128;
constexpr int kSeedBatch = 8;

template <int P>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
    kpool_seed_kernel(const __grid_constant__ KpoolSeedArgs a) {
  __shared__ int32_t s_tok[kWarpsPerCta][kSeedTokensPerWarp];   // token offset in the warp's range
  __shared__ int32_t s_slot[kWarpsPerCta][kSeedTokensPerWarp];  // its tail slot
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t base =
      (static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + warp) * kSeedTokensPerWarp;
  if (base >= a.n_tokens) return;
  const int64_t i0 = base + 4 * lane;
  int32_t t[4], ahead[4];
  const bool vec = (P % 4 == 0) && (reinterpret_cast<uintptr_t>(a.tslot) & 15u) == 0 &&
                   i0 + P + 4 <= a.n_tokens;
  if (vec) {
    const int4 v = *reinterpret_cast<const int4*>(a.tslot + i0);
    const int4 w = *reinterpret_cast<const int4*>(a.tslot + i0 + P);
    t[0] = v.x, t[1] = v.y, t[2] = v.z, t[3] = v.w;
    ahead[0] = w.x, ahead[1] = w.y, ahead[2] = w.z, ahead[3] = w.w;
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      t[q] = i0 + q < a.n_tokens ? a.tslot[i0 + q] : -1;
      ahead[q] = i0 + q + P < a.n_tokens ? a.tslot[i0 + q + P] : -1;
    }
  }
  int n = 0;  // selected tokens so far (warp-uniform)
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    // a negative ahead slot belongs to no block; otherwise compare blocks (t >= 0 here)
    bool tail = t[q] >= 0 && !(ahead[q] >= 0 && ahead[q] / P == t[q] / P);
    if (tail && t[q] / P >= a.num_blocks) {
      flag_error(a.err, CKV_DEVERR_TAIL_BLOCK);
      tail = false;
    }
    const uint32_t m = __ballot_sync(0xFFFFFFFFu, tail);
    if (tail) {
      const int at = n + __popc(m & ((1u << lane) - 1u));
      s_tok[warp][at] = 4 * lane + q;
      s_slot[warp][at] = t[q];
    }
    n += __popc(m);
  }
  __syncwarp();
  // item i of the copy: row i / 64 of the list, array (i / 32) & 1, 8-byte chunk i & 31
  const int items = n * 64;
  for (int c0 = 0; c0 < items; c0 += 32 * kSeedBatch) {
    uint2 v[kSeedBatch];
    uint16_t* dst[kSeedBatch];
#pragma unroll
    for (int u = 0; u < kSeedBatch; ++u) {
      const int i = c0 + 32 * u + lane;
      dst[u] = nullptr;
      if (i < items) {
        const int r = i >> 6, arr = (i >> 5) & 1;
        const int64_t tok = base + s_tok[warp][r];
        const int64_t slot = s_slot[warp][r];
        const uint16_t* src = (arr ? a.score : a.key) + tok * kD + 4 * lane;
        v[u] = ld_stream_u2(src);
        dst[u] = a.ring + (slot / P) * 2 * P * kD + arr * P * kD + (slot % P) * kD + 4 * lane;
      }
    }
#pragma unroll
    for (int u = 0; u < kSeedBatch; ++u)
      if (dst[u]) *reinterpret_cast<uint2*>(dst[u]) = v[u];
  }
}
// Automatic choice: one warp per pool below 65,536 pools, the persistent
// bulk-copy pipeline from there (measured: warp per pool faster by 6-21% up to
// 16,384 pools, equal at 65,536, 3% slower at 262,144).
constexpr int64_t kBulkMinPools = 65536;

template <int P, bool kRound, int W, int S>
cudaError_t compress_bulk(const KpoolCompressArgs& a, bool use_pdl, cudaStream_t s) {
  using L = BulkLayout<P, W, S>;
  auto kern = kpool_compress_bulk_kernel<P, kRound, W, S>;
  cudaError_t e = set_max_smem_once<kpool_compress_bulk_kernel<P, kRound, W, S>>(L::kBytes);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  return launch_ex(kern, dim3(sms), dim3(W * 32), L::kBytes, use_pdl, s, a);
}

// Pool -> token index expansion with the tail appended: one warp per row.  The
// warp copies the row's pool ids into shared memory with one coalesced pass,
// then writes the row's columns four at a time per lane as 16-byte stores (a
// row starts on a 4-byte boundary only, so the columns before its first
// 16-byte boundary and the last ones are written one by one), with no global
// load inside the loop; column -> (pool, offset) uses a shift and a mask when
// P is a power of two, a 32-bit division otherwise.
constexpr int kExpandWarps = 8;
constexpr int kExpandMaxGroups = 2048;  // pool ids per row staged in smem (8 KB per warp)

__global__ void __launch_bounds__(kExpandWarps * 32)
    expand_pools_kernel(const __grid_constant__ ExpandArgs a) {
  extern __shared__ int32_t s_ids[];  // [kExpandWarps][groups]
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t P = static_cast<uint32_t>(a.P);
  const uint32_t G = static_cast<uint32_t>(a.groups);
  const uint32_t gcols = G * P, cols = gcols + P - 1;
  const bool pow2 = (P & (P - 1)) == 0;
  const uint32_t shift = pow2 ? static_cast<uint32_t>(__ffs(static_cast<int>(P)) - 1) : 0u;
  int32_t* ids = s_ids + warp * G;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * kExpandWarps + warp; r < a.rows;
       r += static_cast<int64_t>(gridDim.x) * kExpandWarps) {
    const int32_t* src = a.pool_ids + r * a.stride;
    for (uint32_t g = lane; g < G; g += 32) ids[g] = __ldg(src + g);
    const int64_t s = __ldg(a.seq_lens + r);
    const int64_t tail_start = s - s % static_cast<int64_t>(P);
    const int64_t tail_count = s - tail_start;
    __syncwarp();
    int32_t* dst = a.out + r * cols;
    auto value = [&](uint32_t c) -> int32_t {
      if (c < gcols) {
        const uint32_t g = pow2 ? (c >> shift) : c / P;
        const int64_t id = ids[g];
        return id >= 0 ? static_cast<int32_t>(id * P + (c - g * P)) : -1;
      }
      const int64_t i = c - gcols;
      return i < tail_count ? static_cast<int32_t>(tail_start + i) : -1;
    };
    // columns [0, head) up to the row's first 16-byte boundary, then four per
    // lane per step, then the last (cols - head) % 4
    const uint32_t head = min(cols, ((16u - (static_cast<uint32_t>(reinterpret_cast<uintptr_t>(dst)) & 15u)) & 15u) / 4u);
    if (lane < head) dst[lane] = value(lane);
    const uint32_t nvec = (cols - head) / 4;
    int4* vdst = reinterpret_cast<int4*>(dst + head);
    for (uint32_t v = lane; v < nvec; v += 32) {
      const uint32_t c = head + 4 * v;
      vdst[v] = make_int4(value(c), value(c + 1), value(c + 2), value(c + 3));
    }
    const uint32_t done = head + 4 * nvec;
    if (done + lane < cols) dst[done + lane] = value(done + lane);
    __syncwarp();
  }
}

template <int P>
cudaError_t compress_p(const KpoolCompressArgs& a, bool round_scale, bool use_pdl, cudaStream_t s) {
  const int v = kpool_compress_variant();
  // 8 warps per CTA, each with 3 stages in its ring (measured faster than 12 x 2:
  // more bytes in flight per warp matter more than more warps)
  if (v == 2 || (v == 0 && a.n_pools >= kBulkMinPools))
    return round_scale ? compress_bulk<P, true, 8, 3>(a, use_pdl, s) : compress_bulk<P, false, 8, 3>(a, use_pdl, s);
  const dim3 grid(static_cast<unsigned>((a.n_pools + kWarpsPerCta - 1) / kWarpsPerCta));
  return round_scale
             ? launch_ex(kpool_compress_kernel<P, true>, grid, dim3(kWarpsPerCta * 32), 0, use_pdl, s, a)
             : launch_ex(kpool_compress_kernel<P, false>, grid, dim3(kWarpsPerCta * 32), 0, use_pdl, s, a);
}

template <int P>
cudaError_t decode_p(const KpoolDecodeArgs& a, bool round_scale, bool use_pdl, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>(a.B));
  return round_scale ? launch_ex(kpool_decode_kernel<P, true>, grid, dim3(kDecThreads), 0, use_pdl, s, a)
                     : launch_ex(kpool_decode_kernel<P, false>, grid, dim3(kDecThreads), 0, use_pdl, s, a);
}

template <int P>
cudaError_t seed_p(const KpoolSeedArgs& a, cudaStream_t s) {
  const int64_t per_cta = static_cast<int64_t>(kSeedTokensPerWarp) * kWarpsPerCta;
  const dim3 grid(static_cast<unsigned>((a.n_tokens + per_cta - 1) / per_cta));
  return launch_ex(kpool_seed_kernel<P>, grid, dim3(kWarpsPerCta * 32), 0, false, s, a);
}

}  // namespace

cudaError_t launch_kpool_compress(const KpoolCompressArgs& a, int P, bool round_scale,
                                  bool use_pdl, cudaStream_t s) {
  switch (P) {
    case 1: return compress_p<1>(a, round_scale, use_pdl, s);
    case 2: return compress_p<2>(a, round_scale, use_pdl, s);
    case 4: return compress_p<4>(a, round_scale, use_pdl, s);
    case 8: return compress_p<8>(a, round_scale, use_pdl, s);
    case 16: return compress_p<16>(a, round_scale, use_pdl, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_kpool_decode_update(const KpoolDecodeArgs& a, int P, bool round_scale,
                                       bool use_pdl, cudaStream_t s) {
  switch (P) {
    case 1: return decode_p<1>(a, round_scale, use_pdl, s);
    case 2: return decode_p<2>(a, round_scale, use_pdl, s);
    case 4: return decode_p<4>(a, round_scale, use_pdl, s);
    case 8: return decode_p<8>(a, round_scale, use_pdl, s);
    case 16: return decode_p<16>(a, round_scale, use_pdl, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_expand_pools(const ExpandArgs& a, bool use_pdl, cudaStream_t s) {
  if (a.groups > kExpandMaxGroups) return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(kExpandWarps) * a.groups * sizeof(int32_t);
  cudaError_t e = set_max_smem_once<expand_pools_kernel>(kExpandWarps * kExpandMaxGroups * 4);
  if (e != cudaSuccess) return e;
  const int64_t blocks = (static_cast<int64_t>(a.rows) + kExpandWarps - 1) / kExpandWarps;
  const dim3 grid(static_cast<unsigned>(blocks < (1 << 20) ? blocks : (1 << 20)));
  return launch_ex(expand_pools_kernel, grid, dim3(kExpandWarps * 32), smem, use_pdl, s, a);
}

cudaError_t launch_kpool_seed_tail(const KpoolSeedArgs& a, int P, cudaStream_t s) {
  switch (P) {
    case 1: return seed_p<1>(a, s);
    case 2: return seed_p<2>(a, s);
    case 4: return seed_p<4>(a, s);
    case 8: return seed_p<8>(a, s);
    case 16: return seed_p<16>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ckv
