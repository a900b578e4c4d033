// planner.cpp -- host planner for the online c128 prefill.
//
// Source: sglang page "sgl-project--sglang/.../deepseek_v4/c128_online.cuh",
// plan_online_prefill_host and struct OnlinePrefillPlan.  Request i covers
// global positions [prefix_i, seq_i) with prefix_i = seq_i - extend_i, and
// ragged rows [r_i, r_i + extend_i) with r_i = extend_0 + ... + extend_{i-1}.
// The range is cut at every multiple of 128.  Each piece is described by its
// last token; pieces that end at chunk position 127 close a chunk (compress
// list), the final piece of a request that does not is its trailing partial
// (write list, at most one per request).
#include <cstdint>

#include "ckv_launch.h"

namespace ckv {

ckv_status plan_online_prefill_host(const int64_t* seq_lens, const int64_t* extend_lens,
                                    uint32_t B, uint32_t num_tokens,
                                    ckv_plan_entry* compress_plan, ckv_plan_entry* write_plan,
                                    bool pad_for_graph, uint32_t* num_compress,
                                    uint32_t* num_write) {
  // Validate every length first so that nothing is written for a bad batch.
  uint64_t total = 0;
  for (uint32_t i = 0; i < B; ++i) {
    const int64_t seq = seq_lens[i], ext = extend_lens[i];
    if (ext <= 0 || ext > seq || seq > static_cast<int64_t>(UINT32_MAX)) return CKV_ERR_PLAN;
    total += static_cast<uint64_t>(ext);
  }
  if (total != num_tokens) return CKV_ERR_PLAN;

  uint32_t nc = 0, nw = 0;
  uint64_t ragged_base = 0;
  for (uint32_t i = 0; i < B; ++i) {
    const uint64_t seq = static_cast<uint64_t>(seq_lens[i]);
    const uint64_t prefix = seq - static_cast<uint64_t>(extend_lens[i]);
    for (uint64_t first = prefix; first < seq;) {
      const uint64_t chunk_end = (first / 128 + 1) * 128;  // exclusive
      const uint64_t last = (seq < chunk_end ? seq : chunk_end) - 1;
      ckv_plan_entry e;
      e.ragged_id = static_cast<uint32_t>(ragged_base + (last - prefix));
      e.batch_id = i;
      e.position = static_cast<uint32_t>(last);
      e.window_len = static_cast<uint32_t>(last - first + 1);
      if (last % 128 == 127) {
        if (nc >= num_tokens) return CKV_ERR_PLAN;  // cannot happen when totals agree
        compress_plan[nc++] = e;
      } else {
        if (nw >= num_tokens) return CKV_ERR_PLAN;
        write_plan[nw++] = e;
      }
      first = last + 1;
    }
    ragged_base += static_cast<uint64_t>(extend_lens[i]);
  }
  if (pad_for_graph) {
    const ckv_plan_entry sentinel = {0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu};
    for (uint32_t k = nc; k < num_tokens; ++k) compress_plan[k] = sentinel;
    for (uint32_t k = nw; k < num_tokens; ++k) write_plan[k] = sentinel;
    nc = nw = num_tokens;
  }
  *num_compress = nc;
  *num_write = nw;
  return CKV_OK;
}

}  // namespace ckv
