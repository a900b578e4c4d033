// ckv_launch.h -- argument blocks and launchers behind the C ABI (internal).
//
// Each argument block is passed to its kernel by value as a __grid_constant__
// parameter; the C-ABI layer in capi.cu validates sizes before filling it.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "ckv.h"

namespace ckv {

struct KpoolCompressArgs {
  uint8_t* cache;
  int64_t num_pages;
  int64_t page_size;
  const uint16_t* slot_k;
  const uint16_t* slot_score;
  const float* ape;
  const int64_t* loc;
  const uint8_t* write_mask;
  uint8_t* out_fp8;
  float* out_scale;
  float* tap_x;
  uint16_t* tap_xb;
  uint16_t* tap_yb;
  int32_t* err;
  int64_t n_pools;
  int32_t write_cache;
  int32_t page_shift;  // log2(page_size) when page_size is a power of two, else -1
};

struct KpoolDecodeArgs {
  uint8_t* cache;
  int64_t num_pages;
  int64_t page_size;
  uint16_t* ring;
  int64_t num_blocks;
  const int32_t* tail_slot_mapping;
  const int32_t* slot_mapping;
  const int32_t* positions;
  const uint16_t* key;
  int64_t key_sb, key_st;
  const uint16_t* score;
  int64_t score_sb, score_st;
  const float* ape;
  float* tap_x;
  uint16_t* tap_xb;
  uint16_t* tap_yb;
  int32_t* err;
  int32_t B, N;
};

struct KpoolSeedArgs {
  uint16_t* ring;
  int64_t num_blocks;
  const uint16_t* key;
  const uint16_t* score;
  const int32_t* tslot;
  int64_t n_tokens;
  int32_t* err;
};

struct ExpandArgs {
  const int32_t* pool_ids;
  int64_t stride;
  const int64_t* seq_lens;
  int32_t* out;
  int32_t rows, groups, P;
};

struct C128DecodeArgs {
  float* state;
  int64_t num_slots;
  const void* input;
  float* out;
  const float* ape;
  const int32_t* indices;
  const int32_t* seq_lens;
  int32_t* err;
  int32_t B;
  // optional FP8 output stage (cache == nullptr: none): every output row is
  // also stored into a paged FP8 cache at location cache_loc[row], each
  // 128-channel block bf16-rounded, Hadamard-rotated, bf16-rounded and
  // absmax-quantised with its own fp32 scale
  uint8_t* cache;
  const int64_t* cache_loc;
  int64_t num_pages;
  int32_t page_size;
  int32_t round_scale;
};

struct C128PrefillArgs {
  float* state;
  int64_t num_slots;
  const void* input;
  int64_t num_tokens;
  float* out;
  const float* ape;
  const int32_t* indices;
  const int32_t* load_indices;
  const ckv_plan_entry* compress_plan;
  const ckv_plan_entry* write_plan;
  // nullable: device [2] counts of valid entries (read by the kernels, after
  // the programmatic-dependency wait), clamped to num_compress / num_write
  const uint32_t* counts;
  int32_t* err;
  uint32_t num_compress;
  uint32_t num_write;
  int32_t B;
  // optional FP8 output stage (cache == nullptr: none): every output row is
  // also stored into a paged FP8 cache at location cache_loc[row], each
  // 128-channel block bf16-rounded, Hadamard-rotated, bf16-rounded and
  // absmax-quantised with its own fp32 scale
  uint8_t* cache;
  const int64_t* cache_loc;
  int64_t num_pages;
  int32_t page_size;
  int32_t round_scale;
  // write pass only, set by the launcher when the write launch is a
  // programmatic dependent of this call's own compress launch: everything
  // the write pass reads except the state was final before that launch began,
  // so the kernel waits for its predecessor only before touching the state
  int32_t write_early;
};

cudaError_t launch_kpool_compress(const KpoolCompressArgs& a, int P, bool round_scale,
                                  bool use_pdl, cudaStream_t s);
cudaError_t launch_kpool_decode_update(const KpoolDecodeArgs& a, int P, bool round_scale,
                                       bool use_pdl, cudaStream_t s);
cudaError_t launch_kpool_seed_tail(const KpoolSeedArgs& a, int P, cudaStream_t s);
cudaError_t launch_expand_pools(const ExpandArgs& a, bool use_pdl, cudaStream_t s);
cudaError_t launch_c128_decode(const C128DecodeArgs& a, int D, int in_dtype, bool use_pdl,
                               cudaStream_t s);
cudaError_t launch_c128_prefill(const C128PrefillArgs& a, int D, int in_dtype, bool use_pdl,
                                cudaStream_t s);

// TMA-pipelined compress pass (prefill_tma.cu).
bool c128_prefill_tma_supported(const C128PrefillArgs& a, int D, int in_dtype);
cudaError_t launch_c128_prefill_compress_tma(const C128PrefillArgs& a, int D, int in_dtype,
                                             bool use_pdl, cudaStream_t s);
cudaError_t launch_wait_timeout_selftest(int32_t* err, uint64_t limit_ns, cudaStream_t s);
// 0 auto, 1 one CTA per segment, 2 TMA pipeline (capi.cu).
int prefill_variant();
// 0 auto, 1 one warp per pool, 2 persistent bulk-copy pipeline (capi.cu).
int kpool_compress_variant();

// Device planner (planner_device.cu).
cudaError_t launch_plan_device(const int64_t* seq_lens, const int64_t* extend_lens, uint32_t B,
                               uint32_t num_tokens, ckv_plan_entry* compress_plan,
                               ckv_plan_entry* write_plan, bool pad, uint32_t* counts,
                               int32_t* err, bool use_pdl, cudaStream_t s);

// Host planner (planner.cpp).
ckv_status plan_online_prefill_host(const int64_t* seq_lens, const int64_t* extend_lens,
                                    uint32_t B, uint32_t num_tokens,
                                    ckv_plan_entry* compress_plan, ckv_plan_entry* write_plan,
                                    bool pad_for_graph, uint32_t* num_compress,
                                    uint32_t* num_write);

// validate.cu: clear `bits` (ceil(range / 32) words), then flag repeated or
// out-of-range non-negative ids of the first n (int32 when id_bytes == 4,
// else int64).
cudaError_t launch_check_distinct(const void* ids, int id_bytes, int64_t n, int64_t range, uint32_t* bits,
                                  int32_t* err, cudaStream_t s);

// validate.cu: the same check with the bitmap in a static device array of
// noalloc_check_max_range() bits shared by every call (no allocation).
int64_t noalloc_check_max_range();
cudaError_t launch_check_distinct_noalloc(const void* ids, int id_bytes, int64_t n, int64_t range, int32_t* err,
                                          cudaStream_t s);

// probe.cu: latency floors of a decode-sized launch (hops 0, 1 or 2 dependent
// global round trips per warp).
cudaError_t launch_latency_probe(int hops, const int32_t* idx, const void* rows, int64_t num_rows, void* out,
                                 int32_t n_warps, int32_t warps_per_cta, bool use_pdl, cudaStream_t s);

}  // namespace ckv
