// ckv_oracle.cpp -- plain, slow CPU oracle for gated-softmax KV compression.
//
// TEST INFRASTRUCTURE ONLY.  This file is the independent reference that the
// CUDA library is checked against.  Only the test suite, the smoke check and
// the CPU-baseline leg of the benchmark may load it; the product path never
// links, imports or calls it.  It shares no code, header, table or constant
// generator with the CUDA sources.
//
// Sources (web pages; cited by page title and the routine on it):
//   [KPOOL] "vllm.models.glm5next.amd.ops.kpool_compress" (vLLM docs page):
//           _kpool_decode_update_batched_kernel, _kpool_softmax_rotate_write_cache_kernel,
//           kpool_compress_and_write_cache, kpool_decode_update_and_maybe_write_cache_batched,
//           _kpool_tail_seed_kernel.
//   [C128]  "sgl-project--sglang/.../deepseek_v4/c128_online.cuh" (sglang source page):
//           OnlinePrefillPlan, flash_c128_online_decode, flash_c128_online_prefill,
//           plan_online_prefill_host.
//
// Arithmetic: softmax, sums and merges are done in double, straight from the
// definitions (two-pass softmax over a whole chunk: max, then exp/sum).  The
// steps whose precision the pages fix are done in that precision: the two
// bf16 rounding points of the pooled path, the fp32 Hadamard rotation of a
// bf16 vector, and the fp32 absmax/scale/divide of the FP8 quantisation.
// Readings of points the pages leave open are named where they are used.
//
// Compile with -ffp-contract=off (no fused multiply-add) so results do not
// depend on the host ISA.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#include <thread>
#include <algorithm>
#include <functional>

namespace {

// ---------------------------------------------------------------------------
// Number formats
// ---------------------------------------------------------------------------

// bf16 = the top 16 bits of an IEEE binary32: 1 sign, 8 exponent, 7 stored
// mantissa bits.  Round-to-nearest-even from a double, written from the
// format definition: find the quantum (spacing of bf16 values at |x|) and
// round |x| / quantum to the nearest integer, ties to even.
uint16_t bf16_from_double(double x) {
  if (std::isnan(x)) return 0x7FC0;
  const bool neg = std::signbit(x);
  double a = std::fabs(x);
  uint32_t bits;
  if (a == 0.0) {
    bits = 0;
  } else {
    int e;  // a = f * 2^e, f in [0.5, 1)
    std::frexp(a, &e);
    // Normal bf16 numbers have 8 significant bits; the smallest normal is
    // 2^-126, below which the quantum stays at 2^-133 (subnormals).
    int qexp = std::max(e - 8, -133);
    double r = std::nearbyint(std::ldexp(a, -qexp));  // ties to even (default mode)
    double v = std::ldexp(r, qexp);
    // Largest finite bf16 is (2 - 2^-7) * 2^127; anything that rounds above it is inf.
    const double bf16_max = std::ldexp(255.0, 120);
    if (v > bf16_max) {
      bits = 0x7F800000u;
    } else {
      float f = static_cast<float>(v);  // exact: v has <= 8 significant bits
      std::memcpy(&bits, &f, 4);
    }
  }
  uint16_t h = static_cast<uint16_t>(bits >> 16);
  if (neg) h |= 0x8000;
  return h;
}

float bf16_to_float(uint16_t h) {
  uint32_t bits = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &bits, 4);
  return f;
}

// OCP FP8 E4M3 ("e4m3fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits, no
// infinities, S.1111.111 is NaN, largest finite 1.75 * 2^8 = 448, smallest
// normal 2^-6, subnormals m * 2^-9.  Decode follows the definition.
float e4m3_decode(uint8_t c) {
  const int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
  if (e == 15 && m == 7) return std::nanf("");
  double v = (e == 0) ? std::ldexp(static_cast<double>(m), -9)
                      : std::ldexp(1.0 + m / 8.0, e - 7);
  return static_cast<float>(s ? -v : v);
}

// Encode with round-to-nearest-even and saturation to +-448 (reading: the
// pages store an already clamped fp32 into an FP8 tensor; the FP8 type is the
// OCP e4m3fn one with max 448).  A value that rounds to zero keeps its sign.
uint8_t e4m3_encode(float xf) {
  if (std::isnan(xf)) return 0x7F;
  const double x = xf;
  const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  double a = std::fabs(x);
  if (a >= 448.0) return sign | 0x7E;
  int e;
  std::frexp(a, &e);                  // a in [2^(e-1), 2^e)
  int qexp = std::max(e - 4, -9);     // 4 significant bits; subnormal quantum 2^-9
  double r = std::ldexp(std::nearbyint(std::ldexp(a, -qexp)), qexp);
  if (r == 0.0) return sign;
  if (r >= 448.0) return sign | 0x7E;  // cannot exceed 448 after the test above, kept for clarity
  if (r < std::ldexp(1.0, -6)) {       // subnormal: r = m * 2^-9, m in 1..7
    int m = static_cast<int>(std::ldexp(r, 9));
    return sign | static_cast<uint8_t>(m);
  }
  int er;
  double fr = std::frexp(r, &er);     // r = fr * 2^er, fr in [0.5,1)
  int E = er - 1;                     // r = (2 fr) * 2^E, 2fr in [1,2)
  int m = static_cast<int>((2.0 * fr - 1.0) * 8.0);
  return sign | static_cast<uint8_t>(((E + 7) << 3) | m);
}

// 2^ceil(log2(v)) for a positive finite v, exactly (reading: the pooled path's
// power-of-two scale is the smallest power of two >= v, so a power of two maps
// to itself).
float pow2_ceil(float v) {
  int e;
  double f = std::frexp(static_cast<double>(v), &e);  // v = f * 2^e, f in [0.5, 1)
  if (f == 0.5) return v;                             // already a power of two
  return static_cast<float>(std::ldexp(1.0, e));
}

// ---------------------------------------------------------------------------
// Hadamard-128 rotation.  The pages call `_hadamard128` but do not print it.
// Reading: the Sylvester-ordered Walsh-Hadamard matrix H[i][j] =
// (-1)^popcount(i & j), scaled by 1/sqrt(128) so that the rotation is
// orthonormal and applying it twice gives the identity.
// ---------------------------------------------------------------------------

// Definition: a dense matrix-vector product in double.
void hadamard128_exact(const double* in, double* out) {
  const double c = 1.0 / std::sqrt(128.0);
  for (int i = 0; i < 128; ++i) {
    double acc = 0.0;
    for (int j = 0; j < 128; ++j) {
      const int parity = __builtin_popcount(static_cast<unsigned>(i & j)) & 1;
      acc += parity ? -in[j] : in[j];
    }
    out[i] = acc * c;
  }
}

// The pages apply the rotation to an fp32 tensor, so the rotation itself runs
// in fp32.  Reading of its rounding path: the fast transform with butterfly
// stages of span 1, 2, 4, ..., 64 in that order, each stage forming (u + v,
// u - v) with fp32 round-to-nearest, followed by a single fp32 multiply by
// fp32(1/sqrt(128)).
void hadamard128_fp32(const float* in, float* out) {
  float a[128];
  for (int i = 0; i < 128; ++i) a[i] = in[i];
  for (int h = 1; h < 128; h <<= 1) {
    for (int i = 0; i < 128; ++i) {
      if (i & h) continue;
      const float u = a[i], v = a[i + h];
      a[i] = u + v;
      a[i + h] = u - v;
    }
  }
  const float c = static_cast<float>(1.0 / std::sqrt(128.0));
  for (int i = 0; i < 128; ++i) out[i] = a[i] * c;
}

// Per-vector absmax FP8 quantisation ([KPOOL], the quant block of
// _kpool_softmax_rotate_write_cache_kernel): absmax = max(max|y|, 1e-4);
// scale = round ? 2^ceil(log2(absmax/448)) : absmax/448 (both via an fp32
// multiply by fp32(1/448)); q = e4m3(clamp(y / scale, -448, 448)).
void quantize_row(const uint16_t* yb, int D, int round_scale, uint8_t* q, float* scale_out) {
  float absmax = 0.0f;
  for (int d = 0; d < D; ++d) absmax = std::max(absmax, std::fabs(bf16_to_float(yb[d])));
  absmax = std::max(absmax, 1e-4f);
  const float inv448 = 1.0f / 448.0f;
  const float v = absmax * inv448;
  const float scale = round_scale ? pow2_ceil(v) : v;
  for (int d = 0; d < D; ++d) {
    float t = bf16_to_float(yb[d]) / scale;
    t = std::min(std::max(t, -448.0f), 448.0f);
    q[d] = e4m3_encode(t);
  }
  *scale_out = scale;
}

// Gated softmax over one pool ([KPOOL], passes 1 and 2 of both kernels), the
// plain two-pass definition in double:
//   z_j[d] = score_j[d] + ape_j[d],  x[d] = sum_j e^{z_j - max} k_j / sum_j e^{z_j - max}
// then x -> bf16 -> H128 (fp32) -> bf16 -> absmax FP8.
void pool_compress(const float* k /*[P][D]*/, const float* s /*[P][D]*/, const float* ape,
                   int P, int D, int round_scale, double* x, uint16_t* xb, uint16_t* yb,
                   uint8_t* q, float* scale) {
  for (int d = 0; d < D; ++d) {
    double mx = -INFINITY;
    for (int j = 0; j < P; ++j)
      mx = std::max(mx, static_cast<double>(s[j * D + d]) + ape[j * D + d]);
    double num = 0.0, den = 0.0;
    for (int j = 0; j < P; ++j) {
      const double w = std::exp(static_cast<double>(s[j * D + d]) + ape[j * D + d] - mx);
      den += w;
      num += w * k[j * D + d];
    }
    x[d] = num / den;
    xb[d] = bf16_from_double(x[d]);
  }
  // D == 128 for the rotation (checked by the callers).
  float xf[128], yf[128];
  for (int d = 0; d < 128; ++d) xf[d] = bf16_to_float(xb[d]);
  hadamard128_fp32(xf, yf);
  for (int d = 0; d < 128; ++d) yb[d] = bf16_from_double(yf[d]);
  quantize_row(yb, 128, round_scale, q, scale);
}

// Linear in-page layout of the compressed-K paged cache (reading: the pages'
// `_cache_k_offset` / ROCm preshuffle layout is not defined on them, so every
// page stores its rows as row-major [page_size][D] FP8 bytes followed by
// page_size fp32 scales).
void cache_store(uint8_t* cache, int64_t page_size, int D, int64_t loc, const uint8_t* q, float scale) {
  const int64_t page = loc / page_size, tok = loc % page_size;
  uint8_t* base = cache + page * page_size * (D + 4);
  std::memcpy(base + tok * D, q, D);
  std::memcpy(base + page_size * D + 4 * tok, &scale, 4);
}

void parallel_for(int64_t n, int threads, const std::function<void(int64_t, int64_t)>& fn) {
  if (threads <= 1 || n < 2) {
    fn(0, n);
    return;
  }
  threads = static_cast<int>(std::min<int64_t>(threads, n));
  std::vector<std::thread> pool;
  const int64_t per = (n + threads - 1) / threads;
  for (int t = 0; t < threads; ++t) {
    const int64_t lo = t * per, hi = std::min(n, lo + per);
    if (lo >= hi) break;
    pool.emplace_back(fn, lo, hi);
  }
  for (auto& th : pool) th.join();
}

inline double load_in(const void* p, int dtype, int64_t i) {
  if (dtype == 0) return static_cast<const float*>(p)[i];
  return bf16_to_float(static_cast<const uint16_t*>(p)[i]);
}

}  // namespace

extern "C" {

// ----------------------------- formats ------------------------------------
uint16_t ora_bf16_from_double(double x) { return bf16_from_double(x); }
float ora_bf16_to_float(uint16_t h) { return bf16_to_float(h); }
uint8_t ora_e4m3_encode(float x) { return e4m3_encode(x); }
float ora_e4m3_decode(uint8_t c) { return e4m3_decode(c); }
float ora_pow2_ceil(float v) { return pow2_ceil(v); }
void ora_hadamard128_exact(const double* in, double* out) { hadamard128_exact(in, out); }
void ora_hadamard128_fp32(const float* in, float* out) { hadamard128_fp32(in, out); }
void ora_quantize_row(const uint16_t* yb, int D, int round_scale, uint8_t* q, float* scale) {
  quantize_row(yb, D, round_scale, q, scale);
}
// Rotation stage alone on a bf16 row: yb = bf16(H128_fp32(xb)).
void ora_rotate_bf16(const uint16_t* xb, uint16_t* yb) {
  float xf[128], yf[128];
  for (int d = 0; d < 128; ++d) xf[d] = bf16_to_float(xb[d]);
  hadamard128_fp32(xf, yf);
  for (int d = 0; d < 128; ++d) yb[d] = bf16_from_double(yf[d]);
}

// One pool from fp32 views of bf16 keys/scores (any values allowed).
void ora_pool_compress(const float* k, const float* s, const float* ape, int P, int D, int round_scale,
                       double* x, uint16_t* xb, uint16_t* yb, uint8_t* q, float* scale) {
  pool_compress(k, s, ape, P, D, round_scale, x, xb, yb, q, scale);
}

// ------------------- pooled one-shot compression --------------------------
// [KPOOL] kpool_compress_and_write_cache / _kpool_softmax_rotate_write_cache_kernel.
// slot_k, slot_score: bf16 [n_pools][P][D]; ape fp32 [P][D]; loc int64 [n_pools];
// write_mask (nullable) uint8 [n_pools]; cache uint8 [pages][page_size][D+4]
// (updated in place when write_cache); out_q/out_scale (nullable) receive the
// FP8 row and scale of every pool; x/xb/yb (nullable) receive the stage taps.
void ora_kpool_compress(uint8_t* cache, int64_t num_pages, int64_t page_size,
                        const uint16_t* slot_k, const uint16_t* slot_score, const float* ape,
                        const int64_t* loc, const uint8_t* write_mask, int write_cache,
                        uint8_t* out_q, float* out_scale, int64_t n_pools, int P, int D,
                        int round_scale, double* tap_x, uint16_t* tap_xb, uint16_t* tap_yb,
                        int threads) {
  (void)num_pages;
  parallel_for(n_pools, threads, [&](int64_t lo, int64_t hi) {
    std::vector<float> k(P * D), s(P * D);
    std::vector<double> x(D);
    std::vector<uint16_t> xb(D), yb(D);
    std::vector<uint8_t> q(D);
    for (int64_t r = lo; r < hi; ++r) {
      if (write_mask && !write_mask[r]) continue;  // masked pools write nothing
      for (int i = 0; i < P * D; ++i) {
        k[i] = bf16_to_float(slot_k[r * P * D + i]);
        s[i] = bf16_to_float(slot_score[r * P * D + i]);
      }
      float scale;
      pool_compress(k.data(), s.data(), ape, P, D, round_scale, x.data(), xb.data(), yb.data(),
                    q.data(), &scale);
      if (write_cache) cache_store(cache, page_size, D, loc[r], q.data(), scale);
      if (out_q) std::memcpy(out_q + r * D, q.data(), D);
      if (out_scale) out_scale[r] = scale;
      if (tap_x) std::memcpy(tap_x + r * D, x.data(), D * sizeof(double));
      if (tap_xb) std::memcpy(tap_xb + r * D, xb.data(), D * 2);
      if (tap_yb) std::memcpy(tap_yb + r * D, yb.data(), D * 2);
    }
  });
}

// ---------------- c128 rows through the pooled output stage ----------------
// [C128] compressed rows combined with the [KPOOL] output stage (neither page
// shows the combination; reading): each 128-channel block of an fp32 row is
// one pooled vector -- bf16 (round to nearest even), the Hadamard-128 reading
// above, bf16, absmax FP8 with its own scale -- and the cache generalises the
// pooled layout: per page, page_size rows of D code bytes (block j at bytes
// 128j..), then page_size * (D/128) fp32 scales (row r, block j at r*(D/128)+j).
// Rows with a negative location are skipped.
void ora_c128_rows_to_cache(uint8_t* cache, int64_t page_size, const float* rows, const int64_t* locs,
                            int64_t n, int D, int round_scale) {
  const int blocks = D / 128;
  const int64_t page_bytes = page_size * (D + 4 * blocks);
  for (int64_t r = 0; r < n; ++r) {
    if (locs[r] < 0) continue;
    const int64_t page = locs[r] / page_size, tok = locs[r] % page_size;
    uint8_t* base = cache + page * page_bytes;
    for (int j = 0; j < blocks; ++j) {
      float xf[128], yf[128];
      uint16_t yb[128];
      uint8_t q[128];
      float scale;
      for (int d = 0; d < 128; ++d) xf[d] = bf16_to_float(bf16_from_double(rows[r * D + 128 * j + d]));
      hadamard128_fp32(xf, yf);
      for (int d = 0; d < 128; ++d) yb[d] = bf16_from_double(yf[d]);
      quantize_row(yb, 128, round_scale, q, &scale);
      std::memcpy(base + tok * D + 128 * j, q, 128);
      std::memcpy(base + page_size * D + 4 * (tok * blocks + j), &scale, 4);
    }
  }
}

// ------------------- pooled decode / verify update ------------------------
// [KPOOL] _kpool_decode_update_batched_kernel, written as the ordered
// per-request loop it describes.  Per request b and token t in order:
//   pos_valid   = slot_mapping >= 0 and position >= 0
//   stash_valid = position >= 0 and tail_slot >= 0
//   slot        = max(position, 0) % P            (physical slot == logical slot)
//   block       = max(tail_slot, 0) / P
//   if pos_valid and slot == P-1: compress the pool made of ring slots
//       j != slot of `block` and the current token at `slot`, and write the
//       FP8 row + scale to the cache at slot_mapping;
//   then, if stash_valid, store the token's key and score into ring slot `slot`.
// ring: bf16 [blocks][2][P][D] (half 0 keys, half 1 scores), updated in place.
void ora_kpool_decode_update(uint8_t* cache, int64_t num_pages, int64_t page_size,
                             uint16_t* ring, int64_t num_blocks, const int32_t* tail_slot_mapping,
                             const int32_t* slot_mapping, const int32_t* positions,
                             const uint16_t* key, const uint16_t* score, const float* ape,
                             int B, int N, int P, int D, int round_scale, double* tap_x,
                             uint16_t* tap_xb, uint16_t* tap_yb, int threads) {
  (void)num_pages;
  (void)num_blocks;
  parallel_for(B, threads, [&](int64_t lo, int64_t hi) {
    std::vector<float> k(P * D), s(P * D);
    std::vector<double> x(D);
    std::vector<uint16_t> xb(D), yb(D);
    std::vector<uint8_t> q(D);
    for (int64_t b = lo; b < hi; ++b) {
      for (int t = 0; t < N; ++t) {
        const int64_t idx = b * N + t;
        const int32_t loc = slot_mapping[idx], pos = positions[idx], tslot = tail_slot_mapping[idx];
        const int32_t safe_pos = std::max(pos, 0);
        const bool pos_valid = loc >= 0 && pos >= 0;
        const bool stash_valid = pos >= 0 && tslot >= 0;
        const int slot = safe_pos % P;
        const int64_t block = static_cast<int64_t>(std::max(tslot, 0)) / P;
        uint16_t* kring = ring + block * 2 * P * D;
        uint16_t* sring = kring + P * D;
        const uint16_t* kcur = key + idx * D;
        const uint16_t* scur = score + idx * D;
        if (pos_valid && slot == P - 1) {
          for (int j = 0; j < P; ++j) {
            for (int d = 0; d < D; ++d) {
              k[j * D + d] = bf16_to_float(j == slot ? kcur[d] : kring[j * D + d]);
              s[j * D + d] = bf16_to_float(j == slot ? scur[d] : sring[j * D + d]);
            }
          }
          float scale;
          pool_compress(k.data(), s.data(), ape, P, D, round_scale, x.data(), xb.data(),
                        yb.data(), q.data(), &scale);
          cache_store(cache, page_size, D, loc, q.data(), scale);
          if (tap_x) std::memcpy(tap_x + idx * D, x.data(), D * sizeof(double));
          if (tap_xb) std::memcpy(tap_xb + idx * D, xb.data(), D * 2);
          if (tap_yb) std::memcpy(tap_yb + idx * D, yb.data(), D * 2);
        }
        if (stash_valid) {
          std::memcpy(kring + slot * D, kcur, D * 2);
          std::memcpy(sring + slot * D, scur, D * 2);
        }
      }
    }
  });
}

// ------------------- tail-ring seed from a prefill batch ------------------
// [KPOOL] _kpool_tail_seed_kernel: token i (tail slot t >= 0) is copied into
// ring[t / P][{key, score}][t % P] iff the token P places ahead is past the
// batch, is padding (slot < 0), or lies in a different tail block.
void ora_kpool_seed_tail(uint16_t* ring, int64_t num_blocks, const uint16_t* key,
                         const uint16_t* score, const int32_t* tslot, int64_t n_tokens, int P, int D) {
  (void)num_blocks;
  for (int64_t i = 0; i < n_tokens; ++i) {
    const int64_t t = tslot[i];
    if (t < 0) continue;
    const int64_t blk = t / P;
    const int64_t ahead = (i + P < n_tokens) ? tslot[i + P] : -1;
    if (ahead >= 0 && ahead / P == blk) continue;
    uint16_t* base = ring + blk * 2 * P * D;
    std::memcpy(base + (t % P) * D, key + i * D, D * 2);
    std::memcpy(base + P * D + (t % P) * D, score + i * D, D * 2);
  }
}

// ------------------- pool -> token expansion with tail append --------------
// [KPOOL] expand_pools_and_append_tail: the identity path of
// expand_pools_to_tokens followed by append_tail_to_topk.  For row r with
// sequence length s and pool_len = s / P:
//   columns [0, G*P): column g*P + o holds pool_ids[r][g] * P + o when the pool
//     id is valid, else -1 (reading: a pool id is valid when it is >= 0; the
//     fused routine receives no separate validity mask);
//   columns [G*P, G*P + P - 1): column G*P + i holds pool_len*P + i when
//     i < s - pool_len*P (the tokens of the incomplete trailing pool), else -1.
// Token ids are formed in 64-bit and stored as int32, as the page's casts do.
void ora_expand_pools_and_append_tail(const int32_t* pool_ids, int64_t stride, const int64_t* seq_lens,
                                      int rows, int groups, int P, int32_t* out) {
  const int64_t cols = static_cast<int64_t>(groups) * P + P - 1;
  for (int r = 0; r < rows; ++r) {
    int32_t* o = out + r * cols;
    for (int g = 0; g < groups; ++g) {
      const int64_t id = pool_ids[r * stride + g];
      for (int k = 0; k < P; ++k)
        o[g * P + k] = id >= 0 ? static_cast<int32_t>(id * P + k) : -1;
    }
    const int64_t tail_start = (seq_lens[r] / P) * P;
    const int64_t tail_count = seq_lens[r] - tail_start;
    for (int i = 0; i < P - 1; ++i)
      o[static_cast<int64_t>(groups) * P + i] = i < tail_count ? static_cast<int32_t>(tail_start + i) : -1;
  }
}

// ------------------- online c128 decode -----------------------------------
// [C128] flash_c128_online_decode.  The running state of a slot is
// (max, sum, kv) with kv already normalised, i.e. for the chunk tokens seen so
// far  sum = sum_i e^{z_i - max},  kv = sum_i e^{z_i - max} k_i / sum.
// The new token sits at chunk position p = (seq_len - 1) % 128 with
// z = score + ape[p].  p == 0 starts a new chunk (max = z, sum = 1, kv = k);
// otherwise the token is merged into the slot's state.  p == 127 closes the
// chunk: kv is emitted as the compressed row and the slot is left untouched;
// otherwise the new state is stored.
// state_in: fp32 [num_slots][3][D]; input: [B][2D] (kv | score), fp32 (dtype 0)
// or bf16 (dtype 1); ape fp32 [128][D].  Outputs: out [B][D], new_state
// [B][3][D] (double), closed[B] = 1 when the row was emitted, 0 when the state
// was stored.
void ora_c128_decode(const float* state_in, const void* input, int in_dtype, const float* ape,
                     const int32_t* indices, const int32_t* seq_lens, int B, int D, double* out,
                     double* new_state, int32_t* closed, int threads) {
  parallel_for(B, threads, [&](int64_t lo, int64_t hi) {
    for (int64_t b = lo; b < hi; ++b) {
      const int p = (seq_lens[b] - 1) % 128;
      const float* st = state_in + static_cast<int64_t>(indices[b]) * 3 * D;
      for (int d = 0; d < D; ++d) {
        const double k = load_in(input, in_dtype, b * 2 * D + d);
        const double z = load_in(input, in_dtype, b * 2 * D + D + d) + ape[p * D + d];
        double m, s, kv;
        if (p == 0) {
          m = z;
          s = 1.0;
          kv = k;
        } else {
          const double m1 = st[d], s1 = st[D + d], k1 = st[2 * D + d];
          m = std::max(m1, z);
          const double w1 = s1 * std::exp(m1 - m);
          const double w2 = std::exp(z - m);
          s = w1 + w2;
          kv = (k1 * w1 + k * w2) / s;
        }
        out[b * D + d] = kv;
        new_state[b * 3 * D + d] = m;
        new_state[b * 3 * D + D + d] = s;
        new_state[b * 3 * D + 2 * D + d] = kv;
      }
      closed[b] = (p == 127) ? 1 : 0;
    }
  });
}

// ------------------- online c128 prefill ----------------------------------
// [C128] flash_c128_online_prefill + run_prefill, computed without the plan.
// Request b owns ragged rows [r_b, r_b + extend_b) for global positions
// [seq_b - extend_b, seq_b).  Every 128-chunk the extend touches is handled
// on its own: a two-pass softmax in double over that chunk's extend tokens
// (bias ape[pos % 128]); if the chunk's first extend token is not at chunk
// position 0, the partial (max, sum, kv) stored at slot load_indices[b] is
// merged in.  A chunk whose last extend token is at chunk position 127 emits
// its kv at the ragged row of that token; a trailing partial chunk becomes the
// request's new state (destined for slot indices[b]).
// Outputs: out [num_tokens][D] + out_written [num_tokens] (rows never
// written are left alone); final_state [B][3][D] + state_written [B].
void ora_c128_prefill(const float* state_in, const void* input, int in_dtype, int64_t num_tokens,
                      const float* ape, const int32_t* load_indices, const int64_t* seq_lens,
                      const int64_t* extend_lens, int B, int D, double* out, uint8_t* out_written,
                      double* final_state, int32_t* state_written, int threads) {
  (void)num_tokens;
  std::vector<int64_t> ragged_base(B + 1, 0);
  for (int b = 0; b < B; ++b) ragged_base[b + 1] = ragged_base[b] + extend_lens[b];
  parallel_for(B, threads, [&](int64_t lo, int64_t hi) {
    std::vector<double> z(128);
    for (int64_t b = lo; b < hi; ++b) {
      const int64_t seq = seq_lens[b], ext = extend_lens[b], prefix = seq - ext;
      state_written[b] = 0;
      int64_t pos = prefix;
      while (pos < seq) {
        const int64_t chunk = pos / 128;
        const int64_t first = pos;
        const int64_t last = std::min(seq, chunk * 128 + 128) - 1;  // inclusive
        const int64_t n = last - first + 1;
        const int64_t row0 = ragged_base[b] + (first - prefix);
        const bool starts_mid = (first % 128) != 0;
        const float* prior = state_in + static_cast<int64_t>(load_indices[b]) * 3 * D;
        for (int d = 0; d < D; ++d) {
          double m = -INFINITY;
          for (int64_t j = 0; j < n; ++j) {
            z[j] = load_in(input, in_dtype, (row0 + j) * 2 * D + D + d) +
                   ape[((first + j) % 128) * D + d];
            m = std::max(m, z[j]);
          }
          double s = 0.0, num = 0.0;
          for (int64_t j = 0; j < n; ++j) {
            const double w = std::exp(z[j] - m);
            s += w;
            num += w * load_in(input, in_dtype, (row0 + j) * 2 * D + d);
          }
          double kv = num / s;
          if (starts_mid) {
            const double m1 = prior[d], s1 = prior[D + d], k1 = prior[2 * D + d];
            const double M = std::max(m1, m);
            const double w1 = s1 * std::exp(m1 - M), w2 = s * std::exp(m - M);
            kv = (k1 * w1 + kv * w2) / (w1 + w2);
            s = w1 + w2;
            m = M;
          }
          if (last % 128 == 127) {
            out[(row0 + n - 1) * D + d] = kv;
          } else {
            final_state[b * 3 * D + d] = m;
            final_state[b * 3 * D + D + d] = s;
            final_state[b * 3 * D + 2 * D + d] = kv;
          }
        }
        if (last % 128 == 127) out_written[row0 + n - 1] = 1;
        else state_written[b] = 1;
        pos = last + 1;
      }
    }
  });
}

// ------------------- brute-force segmenter --------------------------------
// Walks every extend token of every request in ragged order and groups
// consecutive tokens of the same request and the same 128-chunk.  Each group
// becomes a 16-byte entry {ragged_id, batch_id, position, window_len} of its
// LAST token ([C128] OnlinePrefillPlan); groups whose last token sits at chunk
// position 127 go to the compress list, the others to the write list.
// Returns 0 on success, -1 if a list would exceed its capacity.
int ora_plan_segments(const int64_t* seq_lens, const int64_t* extend_lens, int B,
                      uint32_t* compress /*[cap][4]*/, uint32_t* write /*[cap][4]*/, int64_t cap,
                      int64_t* num_compress, int64_t* num_write) {
  int64_t nc = 0, nw = 0, ragged = 0;
  for (int b = 0; b < B; ++b) {
    const int64_t prefix = seq_lens[b] - extend_lens[b];
    int64_t len = 0;
    for (int64_t i = 0; i < extend_lens[b]; ++i, ++ragged) {
      const int64_t pos = prefix + i;
      ++len;
      const bool last_of_request = (i == extend_lens[b] - 1);
      const bool last_of_chunk = (pos % 128) == 127;
      if (!(last_of_request || last_of_chunk)) continue;
      uint32_t* dst;
      if (last_of_chunk) {
        if (nc >= cap) return -1;
        dst = compress + 4 * (nc++);
      } else {
        if (nw >= cap) return -1;
        dst = write + 4 * (nw++);
      }
      dst[0] = static_cast<uint32_t>(ragged);
      dst[1] = static_cast<uint32_t>(b);
      dst[2] = static_cast<uint32_t>(pos);
      dst[3] = static_cast<uint32_t>(len);
      len = 0;
    }
  }
  *num_compress = nc;
  *num_write = nw;
  return 0;
}

}  // extern "C"
