// capi.cu -- the extern "C" entry points declared in include/ckv.h.
//
// Every entry point checks its sizes, flags and pointer alignment on the host,
// fills an argument block and enqueues the kernels on the caller's stream.
// Nothing is allocated and nothing synchronises.
#include <algorithm>
#include <atomic>
#include <cstdint>

#include "ckv.h"
#include "ckv_launch.h"

namespace {

thread_local int32_t g_last_cuda_error = 0;
std::atomic<int32_t> g_prefill_variant{0};
std::atomic<int32_t> g_kpool_compress_variant{0};

ckv_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return CKV_OK;
  g_last_cuda_error = static_cast<int32_t>(e);
  // a failed launch also leaves its error pending in the runtime; take it so
  // that it is not reported again by the next call's launch check
  (void)cudaGetLastError();
  return CKV_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// log2(n) for a power of two n > 0, else -1 (lets the kernels split a cache
// location into page and row with a shift instead of a 64-bit division)
int32_t pow2_shift(int64_t n) {
  if (n <= 0 || (n & (n - 1)) != 0) return -1;
  int32_t s = 0;
  while ((int64_t{1} << s) != n) ++s;
  return s;
}
bool pool_size_ok(int32_t P) { return P == 1 || P == 2 || P == 4 || P == 8 || P == 16; }
bool head_dim_ok(int32_t D) { return D == 128 || D == 256 || D == 512; }

}  // namespace

namespace ckv {
int prefill_variant() { return g_prefill_variant.load(std::memory_order_relaxed); }
int kpool_compress_variant() { return g_kpool_compress_variant.load(std::memory_order_relaxed); }
}  // namespace ckv

extern "C" {

int32_t ckv_c128_prefill_set_variant(int32_t variant) {
  if (variant < 0 || variant > 2) return -1;
  return g_prefill_variant.exchange(variant);
}

int32_t ckv_kpool_compress_set_variant(int32_t variant) {
  if (variant < 0 || variant > 2) return -1;
  return g_kpool_compress_variant.exchange(variant);
}

int32_t ckv_abi_version(void) { return 1; }

ckv_status ckv_wait_timeout_selftest(int32_t* err_word, uint32_t limit_us, void* stream) {
  if (!err_word) return CKV_ERR_NULL;
  if (limit_us == 0 || limit_us > 2000000u) return CKV_ERR_SHAPE;
  return cuda_status(ckv::launch_wait_timeout_selftest(err_word, static_cast<uint64_t>(limit_us) * 1000u,
                                                       static_cast<cudaStream_t>(stream)));
}

int32_t ckv_last_cuda_error(void) { return g_last_cuda_error; }

const char* ckv_status_string(ckv_status s) {
  switch (s) {
    case CKV_OK: return "ok";
    case CKV_ERR_NULL: return "a required pointer is NULL";
    case CKV_ERR_SHAPE: return "unsupported or inconsistent size, stride or flag";
    case CKV_ERR_DTYPE: return "unsupported input dtype";
    case CKV_ERR_ALIGN: return "pointer or stride misaligned (16 bytes for row data, element size for index arrays)";
    case CKV_ERR_PLAN: return "planner: invalid lengths, token count or capacity";
    case CKV_ERR_CUDA: return "CUDA runtime error (see ckv_last_cuda_error)";
    default: return "unknown status";
  }
}

ckv_status ckv_kpool_decode_update(uint8_t* kv_cache, int64_t num_pages, int32_t page_size,
                                   uint16_t* tail_ring, int64_t num_tail_blocks,
                                   const int32_t* tail_slot_mapping, const int32_t* slot_mapping,
                                   const int32_t* positions, const uint16_t* key,
                                   int64_t key_stride_b, int64_t key_stride_t,
                                   const uint16_t* score, int64_t score_stride_b,
                                   int64_t score_stride_t, const float* ape, int32_t B, int32_t N,
                                   int32_t P, int32_t D, int32_t round_scale, float* tap_x,
                                   uint16_t* tap_xb, uint16_t* tap_yb, int32_t use_pdl,
                                   int32_t* err_word, void* stream) {
  if (B < 0 || N < 0 || D != 128 || !pool_size_ok(P) || page_size <= 0 || num_pages < 0 ||
      num_tail_blocks < 0)
    return CKV_ERR_SHAPE;
  if (B == 0 || N == 0) return CKV_OK;
  if (!kv_cache || !tail_ring || !tail_slot_mapping || !slot_mapping || !positions || !key ||
      !score || !ape)
    return CKV_ERR_NULL;
  if (key_stride_b < 0 || key_stride_t < 0 || score_stride_b < 0 || score_stride_t < 0)
    return CKV_ERR_SHAPE;
  if (!aligned(kv_cache, 16) || !aligned(tail_ring, 16) || !aligned(key, 16) ||
      !aligned(score, 16) || !aligned(ape, 16) || key_stride_b % 8 || key_stride_t % 8 ||
      score_stride_b % 8 || score_stride_t % 8 || !aligned(tap_x, 16) || !aligned(tap_xb, 8) ||
      !aligned(tap_yb, 8) || !aligned(tail_slot_mapping, 4) || !aligned(slot_mapping, 4) ||
      !aligned(positions, 4) || !aligned(err_word, 4))
    return CKV_ERR_ALIGN;
  ckv::KpoolDecodeArgs a{};
  a.cache = kv_cache;
  a.num_pages = num_pages;
  a.page_size = page_size;
  a.ring = tail_ring;
  a.num_blocks = num_tail_blocks;
  a.tail_slot_mapping = tail_slot_mapping;
  a.slot_mapping = slot_mapping;
  a.positions = positions;
  a.key = key;
  a.key_sb = key_stride_b;
  a.key_st = key_stride_t;
  a.score = score;
  a.score_sb = score_stride_b;
  a.score_st = score_stride_t;
  a.ape = ape;
  a.tap_x = tap_x;
  a.tap_xb = tap_xb;
  a.tap_yb = tap_yb;
  a.err = err_word;
  a.B = B;
  a.N = N;
  return cuda_status(ckv::launch_kpool_decode_update(a, P, round_scale != 0, use_pdl != 0,
                                                     static_cast<cudaStream_t>(stream)));
}

ckv_status ckv_kpool_compress(uint8_t* kv_cache, int64_t num_pages, int32_t page_size,
                              const uint16_t* slot_k, const uint16_t* slot_score, const float* ape,
                              const int64_t* loc, const uint8_t* write_mask, int32_t write_cache,
                              uint8_t* out_fp8, float* out_scale, int64_t n_pools, int32_t P,
                              int32_t D, int32_t round_scale, float* tap_x, uint16_t* tap_xb,
                              uint16_t* tap_yb, int32_t use_pdl, int32_t* err_word, void* stream) {
  if (n_pools < 0 || D != 128 || !pool_size_ok(P)) return CKV_ERR_SHAPE;
  if (!write_cache && !out_fp8) return CKV_ERR_SHAPE;        // nothing requested
  if ((out_fp8 == nullptr) != (out_scale == nullptr)) return CKV_ERR_NULL;
  if (write_mask && out_fp8) return CKV_ERR_SHAPE;           // masked rows have no output
  if (write_cache && (page_size <= 0 || num_pages < 0)) return CKV_ERR_SHAPE;
  if (n_pools == 0) return CKV_OK;
  if (n_pools > (static_cast<int64_t>(INT32_MAX) / 32) * 8) return CKV_ERR_SHAPE;
  if (!slot_k || !slot_score || !ape || (write_cache && (!kv_cache || !loc))) return CKV_ERR_NULL;
  if (!aligned(slot_k, 16) || !aligned(slot_score, 16) || !aligned(ape, 16) ||
      !aligned(kv_cache, 16) || !aligned(out_fp8, 16) || !aligned(tap_x, 16) ||
      !aligned(tap_xb, 8) || !aligned(tap_yb, 8) || !aligned(loc, 8) || !aligned(out_scale, 4) ||
      !aligned(err_word, 4))
    return CKV_ERR_ALIGN;
  ckv::KpoolCompressArgs a{};
  a.cache = kv_cache;
  a.num_pages = num_pages;
  a.page_size = page_size > 0 ? page_size : 1;
  a.page_shift = pow2_shift(a.page_size);
  a.slot_k = slot_k;
  a.slot_score = slot_score;
  a.ape = ape;
  a.loc = loc;
  a.write_mask = write_mask;
  a.out_fp8 = out_fp8;
  a.out_scale = out_scale;
  a.tap_x = tap_x;
  a.tap_xb = tap_xb;
  a.tap_yb = tap_yb;
  a.err = err_word;
  a.n_pools = n_pools;
  a.write_cache = write_cache != 0;
  return cuda_status(ckv::launch_kpool_compress(a, P, round_scale != 0, use_pdl != 0,
                                                static_cast<cudaStream_t>(stream)));
}

ckv_status ckv_kpool_seed_tail(uint16_t* tail_ring, int64_t num_tail_blocks, const uint16_t* key,
                               const uint16_t* score, const int32_t* tslot, int64_t n_tokens,
                               int32_t P, int32_t D, int32_t* err_word, void* stream) {
  if (n_tokens < 0 || num_tail_blocks < 0 || D != 128 || !pool_size_ok(P)) return CKV_ERR_SHAPE;
  if (n_tokens == 0) return CKV_OK;
  if (n_tokens > (static_cast<int64_t>(INT32_MAX) / 32) * 8) return CKV_ERR_SHAPE;
  if (!tail_ring || !key || !score || !tslot) return CKV_ERR_NULL;
  if (!aligned(tail_ring, 16) || !aligned(key, 16) || !aligned(score, 16) || !aligned(tslot, 4) ||
      !aligned(err_word, 4))
    return CKV_ERR_ALIGN;
  ckv::KpoolSeedArgs a{};
  a.ring = tail_ring;
  a.num_blocks = num_tail_blocks;
  a.key = key;
  a.score = score;
  a.tslot = tslot;
  a.n_tokens = n_tokens;
  a.err = err_word;
  return cuda_status(ckv::launch_kpool_seed_tail(a, P, static_cast<cudaStream_t>(stream)));
}

ckv_status ckv_expand_pools_and_append_tail(const int32_t* pool_ids, int64_t pool_ids_stride,
                                           const int64_t* seq_lens, int32_t rows, int32_t n_groups,
                                           int32_t P, int32_t* out, int32_t use_pdl, void* stream) {
  if (rows < 0 || n_groups < 0 || n_groups > 2048 || P < 1 || P > 1024 || pool_ids_stride < n_groups)
    return CKV_ERR_SHAPE;
  const int64_t cols = static_cast<int64_t>(n_groups) * P + P - 1;
  if (rows == 0 || cols == 0) return CKV_OK;
  if (cols > static_cast<int64_t>(INT32_MAX) - 256) return CKV_ERR_SHAPE;
  if (!seq_lens || !out || (n_groups > 0 && !pool_ids)) return CKV_ERR_NULL;
  if (!aligned(pool_ids, 4) || !aligned(seq_lens, 8) || !aligned(out, 4)) return CKV_ERR_ALIGN;
  ckv::ExpandArgs a{};
  a.pool_ids = pool_ids;
  a.stride = pool_ids_stride;
  a.seq_lens = seq_lens;
  a.out = out;
  a.rows = rows;
  a.groups = n_groups;
  a.P = P;
  return cuda_status(ckv::launch_expand_pools(a, use_pdl != 0, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// The optional FP8 output stage of the c128 calls (kv_cache == nullptr: none).
struct Fp8Out {
  uint8_t* kv_cache;
  int64_t num_pages;
  int32_t page_size;
  const int64_t* cache_loc;
  int32_t round_scale;
};

ckv_status fp8_check(const Fp8Out* f) {
  if (!f) return CKV_OK;
  if (f->page_size <= 0 || f->num_pages < 0) return CKV_ERR_SHAPE;
  if (!f->kv_cache || !f->cache_loc) return CKV_ERR_NULL;
  if (!aligned(f->kv_cache, 16) || !aligned(f->cache_loc, 8)) return CKV_ERR_ALIGN;
  return CKV_OK;
}

template <typename Args>
void fp8_set(Args& a, const Fp8Out* f) {
  if (!f) return;
  a.cache = f->kv_cache;
  a.cache_loc = f->cache_loc;
  a.num_pages = f->num_pages;
  a.page_size = f->page_size;
  a.round_scale = f->round_scale;
}

ckv_status c128_decode_impl(float* state, int64_t num_slots, const void* input, ckv_dtype in_dtype, float* out,
                            const float* ape, const int32_t* indices, const int32_t* seq_lens, int32_t B,
                            int32_t D, const Fp8Out* fp8, int32_t use_pdl, int32_t* err_word, void* stream) {
  if (B < 0 || num_slots < 0 || !head_dim_ok(D)) return CKV_ERR_SHAPE;
  if (in_dtype != CKV_F32 && in_dtype != CKV_BF16) return CKV_ERR_DTYPE;
  if (ckv_status c = fp8_check(fp8)) return c;
  if (B == 0) return CKV_OK;
  if (!state || !input || !ape || !indices || !seq_lens || (!out && !fp8)) return CKV_ERR_NULL;
  if (!aligned(state, 16) || !aligned(input, 16) || !aligned(out, 16) || !aligned(ape, 16) ||
      !aligned(indices, 4) || !aligned(seq_lens, 4) || !aligned(err_word, 4))
    return CKV_ERR_ALIGN;
  ckv::C128DecodeArgs a{};
  a.state = state;
  a.num_slots = num_slots;
  a.input = input;
  a.out = out;
  a.ape = ape;
  a.indices = indices;
  a.seq_lens = seq_lens;
  a.err = err_word;
  a.B = B;
  fp8_set(a, fp8);
  return cuda_status(ckv::launch_c128_decode(a, D, in_dtype, use_pdl != 0,
                                             static_cast<cudaStream_t>(stream)));
}

ckv_status c128_prefill_impl(float* state, int64_t num_slots, const void* input, ckv_dtype in_dtype,
                             int64_t num_tokens, float* out, const float* ape, const int32_t* indices,
                             const int32_t* load_indices, int32_t B, const ckv_plan_entry* compress_plan,
                             uint32_t num_compress, const ckv_plan_entry* write_plan, uint32_t num_write,
                             int32_t D, const Fp8Out* fp8, int32_t use_pdl, int32_t* err_word, void* stream) {
  if (B < 0 || num_slots < 0 || num_tokens < 0 || num_tokens > static_cast<int64_t>(UINT32_MAX) ||
      !head_dim_ok(D))
    return CKV_ERR_SHAPE;
  if (in_dtype != CKV_F32 && in_dtype != CKV_BF16) return CKV_ERR_DTYPE;
  if (ckv_status c = fp8_check(fp8)) return c;
  if (num_compress == 0 && num_write == 0) return CKV_OK;
  const uint64_t S = static_cast<uint64_t>(D / 128);
  if (static_cast<uint64_t>(num_compress) * S > static_cast<uint64_t>(INT32_MAX) ||
      static_cast<uint64_t>(num_write) * S > static_cast<uint64_t>(INT32_MAX))
    return CKV_ERR_SHAPE;
  if (!state || !input || !ape || !indices) return CKV_ERR_NULL;
  if ((num_compress && (!compress_plan || (!out && !fp8))) || (num_write && !write_plan)) return CKV_ERR_NULL;
  if (!aligned(state, 16) || !aligned(input, 16) || !aligned(out, 16) || !aligned(ape, 16) ||
      !aligned(compress_plan, 16) || !aligned(write_plan, 16) || !aligned(indices, 4) ||
      !aligned(load_indices, 4) || !aligned(err_word, 4))
    return CKV_ERR_ALIGN;
  ckv::C128PrefillArgs a{};
  a.state = state;
  a.num_slots = num_slots;
  a.input = input;
  a.num_tokens = num_tokens;
  a.out = out;
  a.ape = ape;
  a.indices = indices;
  a.load_indices = load_indices ? load_indices : indices;
  a.compress_plan = compress_plan;
  a.write_plan = write_plan;
  a.err = err_word;
  a.num_compress = num_compress;
  a.num_write = num_write;
  a.B = B;
  fp8_set(a, fp8);
  return cuda_status(ckv::launch_c128_prefill(a, D, in_dtype, use_pdl != 0,
                                              static_cast<cudaStream_t>(stream)));
}

ckv_status c128_prefill_counted_impl(float* state, int64_t num_slots, const void* input, ckv_dtype in_dtype,
                                     int64_t num_tokens, float* out, const float* ape, const int32_t* indices,
                                     const int32_t* load_indices, int32_t B, const ckv_plan_entry* compress_plan,
                                     const ckv_plan_entry* write_plan, const uint32_t* counts, int32_t D,
                                     const Fp8Out* fp8, int32_t use_pdl, int32_t* err_word, void* stream) {
  if (B < 0 || num_slots < 0 || num_tokens < 0 || num_tokens > static_cast<int64_t>(UINT32_MAX) ||
      !head_dim_ok(D))
    return CKV_ERR_SHAPE;
  if (in_dtype != CKV_F32 && in_dtype != CKV_BF16) return CKV_ERR_DTYPE;
  if (ckv_status c = fp8_check(fp8)) return c;
  if (num_tokens == 0 || B == 0) return CKV_OK;
  // every compress segment closes a chunk: per request at most extend/128 + 1 of
  // them, so at most num_tokens/128 + B in total; at most one write segment each
  const uint64_t max_c = std::min<uint64_t>(static_cast<uint64_t>(num_tokens) / 128 + B,
                                            static_cast<uint64_t>(num_tokens));
  const uint64_t max_w = std::min<uint64_t>(B, static_cast<uint64_t>(num_tokens));
  const uint64_t S = static_cast<uint64_t>(D / 128);
  if (max_c * S > static_cast<uint64_t>(INT32_MAX)) return CKV_ERR_SHAPE;
  if (!state || !input || !ape || !indices || (!out && !fp8) || !compress_plan || !write_plan || !counts)
    return CKV_ERR_NULL;
  if (!aligned(state, 16) || !aligned(input, 16) || !aligned(out, 16) || !aligned(ape, 16) ||
      !aligned(compress_plan, 16) || !aligned(write_plan, 16) || !aligned(counts, 4) ||
      !aligned(indices, 4) || !aligned(load_indices, 4) || !aligned(err_word, 4))
    return CKV_ERR_ALIGN;
  ckv::C128PrefillArgs a{};
  a.state = state;
  a.num_slots = num_slots;
  a.input = input;
  a.num_tokens = num_tokens;
  a.out = out;
  a.ape = ape;
  a.indices = indices;
  a.load_indices = load_indices ? load_indices : indices;
  a.compress_plan = compress_plan;
  a.write_plan = write_plan;
  a.counts = counts;
  a.err = err_word;
  a.num_compress = static_cast<uint32_t>(max_c);
  a.num_write = static_cast<uint32_t>(max_w);
  a.B = B;
  fp8_set(a, fp8);
  return cuda_status(ckv::launch_c128_prefill(a, D, in_dtype, use_pdl != 0,
                                              static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

ckv_status ckv_c128_online_decode(float* state, int64_t num_slots, const void* input,
                                  ckv_dtype in_dtype, float* out, const float* ape,
                                  const int32_t* indices, const int32_t* seq_lens, int32_t B,
                                  int32_t D, int32_t use_pdl, int32_t* err_word, void* stream) {
  return c128_decode_impl(state, num_slots, input, in_dtype, out, ape, indices, seq_lens, B, D, nullptr, use_pdl,
                          err_word, stream);
}

ckv_status ckv_c128_online_decode_fp8(float* state, int64_t num_slots, const void* input,
                                      ckv_dtype in_dtype, float* out, const float* ape,
                                      const int32_t* indices, const int32_t* seq_lens, int32_t B,
                                      int32_t D, uint8_t* kv_cache, int64_t num_pages,
                                      int32_t page_size, const int64_t* cache_loc,
                                      int32_t round_scale, int32_t use_pdl, int32_t* err_word,
                                      void* stream) {
  const Fp8Out f{kv_cache, num_pages, page_size, cache_loc, round_scale};
  return c128_decode_impl(state, num_slots, input, in_dtype, out, ape, indices, seq_lens, B, D, &f, use_pdl,
                          err_word, stream);
}

ckv_status ckv_c128_online_prefill(float* state, int64_t num_slots, const void* input,
                                   ckv_dtype in_dtype, int64_t num_tokens, float* out,
                                   const float* ape, const int32_t* indices,
                                   const int32_t* load_indices, int32_t B,
                                   const ckv_plan_entry* compress_plan, uint32_t num_compress,
                                   const ckv_plan_entry* write_plan, uint32_t num_write, int32_t D,
                                   int32_t use_pdl, int32_t* err_word, void* stream) {
  return c128_prefill_impl(state, num_slots, input, in_dtype, num_tokens, out, ape, indices, load_indices, B,
                           compress_plan, num_compress, write_plan, num_write, D, nullptr, use_pdl, err_word,
                           stream);
}

ckv_status ckv_c128_online_prefill_fp8(float* state, int64_t num_slots, const void* input,
                                       ckv_dtype in_dtype, int64_t num_tokens, float* out,
                                       const float* ape, const int32_t* indices,
                                       const int32_t* load_indices, int32_t B,
                                       const ckv_plan_entry* compress_plan, uint32_t num_compress,
                                       const ckv_plan_entry* write_plan, uint32_t num_write,
                                       int32_t D, uint8_t* kv_cache, int64_t num_pages,
                                       int32_t page_size, const int64_t* cache_loc,
                                       int32_t round_scale, int32_t use_pdl, int32_t* err_word,
                                       void* stream) {
  const Fp8Out f{kv_cache, num_pages, page_size, cache_loc, round_scale};
  return c128_prefill_impl(state, num_slots, input, in_dtype, num_tokens, out, ape, indices, load_indices, B,
                           compress_plan, num_compress, write_plan, num_write, D, &f, use_pdl, err_word, stream);
}

ckv_status ckv_c128_online_prefill_counted(float* state, int64_t num_slots, const void* input,
                                           ckv_dtype in_dtype, int64_t num_tokens, float* out,
                                           const float* ape, const int32_t* indices,
                                           const int32_t* load_indices, int32_t B,
                                           const ckv_plan_entry* compress_plan,
                                           const ckv_plan_entry* write_plan, const uint32_t* counts,
                                           int32_t D, int32_t use_pdl, int32_t* err_word,
                                           void* stream) {
  return c128_prefill_counted_impl(state, num_slots, input, in_dtype, num_tokens, out, ape, indices, load_indices,
                                   B, compress_plan, write_plan, counts, D, nullptr, use_pdl, err_word, stream);
}

ckv_status ckv_c128_online_prefill_counted_fp8(float* state, int64_t num_slots, const void* input,
                                               ckv_dtype in_dtype, int64_t num_tokens, float* out,
                                               const float* ape, const int32_t* indices,
                                               const int32_t* load_indices, int32_t B,
                                               const ckv_plan_entry* compress_plan,
                                               const ckv_plan_entry* write_plan,
                                               const uint32_t* counts, int32_t D, uint8_t* kv_cache,
                                               int64_t num_pages, int32_t page_size,
                                               const int64_t* cache_loc, int32_t round_scale,
                                               int32_t use_pdl, int32_t* err_word, void* stream) {
  const Fp8Out f{kv_cache, num_pages, page_size, cache_loc, round_scale};
  return c128_prefill_counted_impl(state, num_slots, input, in_dtype, num_tokens, out, ape, indices, load_indices,
                                   B, compress_plan, write_plan, counts, D, &f, use_pdl, err_word, stream);
}

ckv_status ckv_plan_online_prefill_device(const int64_t* seq_lens, const int64_t* extend_lens,
                                          uint32_t B, uint32_t num_tokens,
                                          ckv_plan_entry* compress_plan, ckv_plan_entry* write_plan,
                                          int32_t pad_for_graph, uint32_t* counts, int32_t use_pdl,
                                          int32_t* err_word, void* stream) {
  if (B > 8192) return CKV_ERR_SHAPE;
  if (!counts) return CKV_ERR_NULL;
  if (B > 0 && (!seq_lens || !extend_lens)) return CKV_ERR_NULL;
  if (num_tokens > 0 && (!compress_plan || !write_plan)) return CKV_ERR_NULL;
  if (!aligned(compress_plan, 16) || !aligned(write_plan, 16) || !aligned(counts, 4) ||
      !aligned(seq_lens, 8) || !aligned(extend_lens, 8) || !aligned(err_word, 4))
    return CKV_ERR_ALIGN;
  return cuda_status(ckv::launch_plan_device(seq_lens, extend_lens, B, num_tokens, compress_plan,
                                             write_plan, pad_for_graph != 0, counts, err_word,
                                             use_pdl != 0, static_cast<cudaStream_t>(stream)));
}

ckv_status ckv_plan_online_prefill(const int64_t* seq_lens, const int64_t* extend_lens, uint32_t B,
                                   uint32_t num_tokens, ckv_plan_entry* compress_plan,
                                   ckv_plan_entry* write_plan, int32_t pad_for_graph,
                                   uint32_t* num_compress, uint32_t* num_write) {
  if (!num_compress || !num_write) return CKV_ERR_NULL;
  if (B > 0 && (!seq_lens || !extend_lens)) return CKV_ERR_NULL;
  if (num_tokens > 0 && (!compress_plan || !write_plan)) return CKV_ERR_NULL;
  return ckv::plan_online_prefill_host(seq_lens, extend_lens, B, num_tokens, compress_plan,
                                       write_plan, pad_for_graph != 0, num_compress, num_write);
}

ckv_status ckv_check_distinct(const void* ids, int32_t id_bytes, int64_t n, int64_t range,
                              uint32_t* scratch, int64_t scratch_words, int32_t* err_word,
                              void* stream) {
  if ((id_bytes != 4 && id_bytes != 8) || n < 0 || range < 1 || range > (int64_t{1} << 40))
    return CKV_ERR_SHAPE;
  if (scratch_words < (range + 31) / 32) return CKV_ERR_SHAPE;
  if (!scratch || !err_word || (n > 0 && !ids)) return CKV_ERR_NULL;
  if (!aligned(ids, static_cast<uintptr_t>(id_bytes)) || !aligned(scratch, 4) || !aligned(err_word, 4))
    return CKV_ERR_ALIGN;
  return cuda_status(ckv::launch_check_distinct(ids, id_bytes, n, range, scratch, err_word,
                                                static_cast<cudaStream_t>(stream)));
}

ckv_status ckv_check_distinct_noalloc(const void* ids, int32_t id_bytes, int64_t n, int64_t range,
                                      int32_t* err_word, void* stream) {
  if ((id_bytes != 4 && id_bytes != 8) || n < 0 || range < 1) return CKV_ERR_SHAPE;
  if (range > ckv::noalloc_check_max_range()) return CKV_ERR_SHAPE;  // beyond the fixed bitmap
  if (!err_word || (n > 0 && !ids)) return CKV_ERR_NULL;
  if (!aligned(ids, static_cast<uintptr_t>(id_bytes)) || !aligned(err_word, 4)) return CKV_ERR_ALIGN;
  return cuda_status(ckv::launch_check_distinct_noalloc(ids, id_bytes, n, range, err_word,
                                                        static_cast<cudaStream_t>(stream)));
}

ckv_status ckv_latency_probe(int32_t hops, const int32_t* idx, const void* rows, int64_t num_rows, void* out,
                             int32_t n_warps, int32_t warps_per_cta, int32_t use_pdl, void* stream) {
  if (hops < 0 || hops > 4 || n_warps < 1 || n_warps > (1 << 30) || warps_per_cta < 1 || warps_per_cta > 32 ||
      num_rows < 0)
    return CKV_ERR_SHAPE;
  if (hops == 3 && (n_warps < 16 || num_rows < 9)) return CKV_ERR_SHAPE;
  if (hops == 4 && (n_warps < 16 || num_rows < 64)) return CKV_ERR_SHAPE;
  if (hops >= 1 && (!idx || !out)) return CKV_ERR_NULL;
  if (hops >= 2 && !rows) return CKV_ERR_NULL;
  if (!aligned(idx, 4) || !aligned(rows, 8) || !aligned(out, 8)) return CKV_ERR_ALIGN;
  return cuda_status(ckv::launch_latency_probe(hops, idx, rows, num_rows, out, n_warps, warps_per_cta,
                                               use_pdl != 0, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
