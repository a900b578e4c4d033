/*
 * ckv.h -- C ABI of the gated-softmax KV compression library (GB300, sm_103a).
 *
 * The method: tokens are grouped into chunks of P consecutive positions and
 * every channel d of a chunk's compressed key is
 *
 *     out[d] = sum_j softmax_j(score_j[d] + ape[j mod P][d]) * k_j[d]
 *
 * (a per-channel softmax over the chunk's tokens).  Two families of calls:
 *   - pooled, P = 16 (or 1, 2, 4, 8), D = 128, bf16 keys/scores: the pooled row
 *     is rounded to bf16, rotated by a 128-point Hadamard transform, rounded
 *     to bf16 again and stored as FP8-e4m3 with one fp32 absmax scale in a
 *     paged cache.  Source: vLLM page "vllm.models.glm5next.amd.ops.kpool_compress".
 *   - online, P = 128, D in {128, 256, 512}, fp32 or bf16 inputs: a per-slot
 *     fp32 running state (max, sum, kv) is updated one token at a time
 *     (decode) or one segment at a time (prefill).  Source: sglang page
 *     "sgl-project--sglang/.../jit_kernel/csrc/deepseek_v4/c128_online.cuh".
 *
 * Conventions for every call below:
 *   - Pointers marked "device" are CUDA device memory owned by the caller;
 *     "host" pointers are ordinary (or pinned) host memory.  The library
 *     allocates nothing and never synchronises the stream.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *     only enqueued; results are visible after the stream reaches it.
 *   - Sizes are checked on the host before anything is launched; a failed
 *     check returns a nonzero ckv_status and launches nothing.  An empty
 *     batch returns CKV_OK and launches nothing.
 *   - `err_word` (device, nullable) receives, by atomic OR, a CKV_DEVERR_*
 *     bit when a kernel meets an index that is out of range (a slot, a tail
 *     block, a cache location, a malformed plan entry).  The offending
 *     access is skipped, never performed; everything else proceeds.  The
 *     word is never cleared by the library.
 *   - Caller contract inherited from the sources: within one call, distinct
 *     requests use distinct tail blocks, state slots and cache locations
 *     (concurrent CTAs touch disjoint memory).  Overlapping calls on
 *     different streams that share buffers race.
 */
#ifndef CKV_H_
#define CKV_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t ckv_status;
#define CKV_OK 0
#define CKV_ERR_NULL 1       /* a required pointer is NULL */
#define CKV_ERR_SHAPE 2      /* unsupported or inconsistent size, stride or flag */
#define CKV_ERR_DTYPE 3      /* unsupported input dtype */
#define CKV_ERR_ALIGN 4      /* a pointer or stride is misaligned: 16 bytes for row data, the element size for index arrays and err_word */
#define CKV_ERR_PLAN 5       /* planner: bad lengths, token count or capacity */
#define CKV_ERR_CUDA 6       /* a CUDA runtime call failed (see ckv_last_cuda_error) */

/* Bits OR-ed into err_word by the kernels (the access is skipped). */
#define CKV_DEVERR_SLOT 0x1u       /* state slot index outside [0, num_slots) */
#define CKV_DEVERR_TAIL_BLOCK 0x2u /* tail block outside [0, num_tail_blocks) */
#define CKV_DEVERR_CACHE_LOC 0x4u  /* cache location outside [0, num_pages * page_size) */
#define CKV_DEVERR_PLAN 0x8u       /* plan entry fields inconsistent or out of range */
#define CKV_DEVERR_SEQ_LEN 0x10u   /* decode seq_len < 1 */
#define CKV_DEVERR_TIMEOUT 0x20u   /* a pipeline wait gave up after 2 s (never expected) */
#define CKV_DEVERR_DISTINCT 0x40u  /* ckv_check_distinct: an id repeats or is >= range */

typedef int32_t ckv_dtype;
#define CKV_F32 0
#define CKV_BF16 1

/* One prefill segment: a run of tokens of one request inside one 128-chunk,
 * described by its LAST token (sglang page, struct OnlinePrefillPlan):
 *   ragged_id  row of the last token in the ragged [num_tokens, 2D] input
 *   batch_id   request index (into indices / load_indices)
 *   position   global position of the last token; position % 128 == 127 for
 *              a compress (chunk-closing) segment, < 127 for a write segment
 *   window_len number of tokens, 1..128; the first token is at ragged row
 *              ragged_id - window_len + 1 and position position - window_len + 1
 * An entry with all four fields 0xFFFFFFFF is a sentinel and is skipped. */
typedef struct ckv_plan_entry {
  uint32_t ragged_id;
  uint32_t batch_id;
  uint32_t position;
  uint32_t window_len;
} ckv_plan_entry;

/* Returns a static, human-readable description of a status code. */
const char* ckv_status_string(ckv_status s);

/* The cudaError_t of the most recent CKV_ERR_CUDA on the calling thread. */
int32_t ckv_last_cuda_error(void);

/* ABI version of this header (incremented on incompatible changes). */
int32_t ckv_abi_version(void);

/*
 * Self-test of the bounded pipeline waits: launches one thread that waits on
 * an mbarrier nothing will ever complete, with a limit of limit_us
 * microseconds (1 .. 2,000,000).  The wait must give up and OR
 * CKV_DEVERR_TIMEOUT into err_word (device int32); the context stays usable.
 * The kernels' own waits use the same code with a two-second limit.
 */
ckv_status ckv_wait_timeout_selftest(int32_t* err_word, uint32_t limit_us, void* stream);

/*
 * Pooled decode / speculative-verify update (vLLM kpool_compress page,
 * _kpool_decode_update_batched_kernel and
 * kpool_decode_update_and_maybe_write_cache_batched).
 *
 * For each request b (processed independently) and each of its N tokens t in
 * order, with idx = b*N + t:
 *   pos_valid   = slot_mapping[idx] >= 0 && positions[idx] >= 0
 *   stash_valid = positions[idx] >= 0 && tail_slot_mapping[idx] >= 0
 *   slot        = max(positions[idx], 0) % P;  block = max(tail_slot_mapping[idx], 0) / P
 *   If pos_valid and slot == P-1 the pool closes: the P tokens are ring slots
 *   0..P-2 of `block` plus the current token, and the compressed FP8 row and
 *   scale are written to the cache at location slot_mapping[idx].  Then, if
 *   stash_valid, the token's key and score are stored in ring slot `slot`
 *   (after the completion read, so a pool sees tokens stashed earlier in the
 *   same call).
 *
 * kv_cache          device uint8 [num_pages][page_size][D+4]: per page,
 *                   page_size rows of D FP8-e4m3 bytes (row-major), then
 *                   page_size fp32 scales.  Location loc is page loc/page_size,
 *                   row loc%page_size.
 * tail_ring         device bf16 [num_tail_blocks][2][P][D]: half 0 keys,
 *                   half 1 gate scores; updated in place.
 * tail_slot_mapping, slot_mapping, positions
 *                   device int32 [B][N]; -1 marks padding.  slot_mapping is
 *                   pool-granular (>= 0 only on a pool's last token).
 * key, score        device bf16, row (b, t) at b*stride_b + t*stride_t
 *                   elements, D contiguous; 16-byte aligned rows.
 * ape               device fp32 [P][D] contiguous (per-slot position bias).
 * P                 1, 2, 4, 8 or 16.  D must be 128.
 * round_scale       nonzero: scale = 2^ceil(log2(absmax/448)); zero: absmax/448.
 * tap_x, tap_xb, tap_yb
 *                   device, nullable, [B*N][D]: the fp32 pooled row, its bf16
 *                   rounding and the bf16 rotated row of every closing token
 *                   (row idx); rows of other tokens are not written.
 * use_pdl           nonzero: launch as a programmatic dependent launch (the kernel
 *                   waits for the preceding grid before it touches memory).
 */
ckv_status ckv_kpool_decode_update(uint8_t* kv_cache, int64_t num_pages, int32_t page_size,
                                   uint16_t* tail_ring, int64_t num_tail_blocks,
                                   const int32_t* tail_slot_mapping, const int32_t* slot_mapping,
                                   const int32_t* positions, const uint16_t* key,
                                   int64_t key_stride_b, int64_t key_stride_t,
                                   const uint16_t* score, int64_t score_stride_b,
                                   int64_t score_stride_t, const float* ape, int32_t B, int32_t N,
                                   int32_t P, int32_t D, int32_t round_scale, float* tap_x,
                                   uint16_t* tap_xb, uint16_t* tap_yb, int32_t use_pdl,
                                   int32_t* err_word, void* stream);

/*
 * One-shot pooled compression (vLLM kpool_compress page,
 * _kpool_softmax_rotate_write_cache_kernel and kpool_compress_and_write_cache).
 *
 * slot_k, slot_score device bf16 [n_pools][P][D] contiguous.
 * ape                device fp32 [P][D].
 * loc                device int64 [n_pools]: cache location of each pool
 *                    (used only when write_cache != 0).
 * write_mask         device uint8 [n_pools], nullable: pools with 0 write
 *                    nothing (only allowed with out_fp8 == NULL).
 * write_cache        nonzero: store rows + scales into kv_cache (layout as above).
 * out_fp8, out_scale device, nullable together: [n_pools][D] FP8 codes and
 *                    [n_pools] fp32 scales of every pool ("return compressed").
 * At least one of write_cache / out_fp8 must be requested.
 * tap_x, tap_xb, tap_yb: device, nullable, [n_pools][D] stage taps.
 * use_pdl            as for ckv_kpool_decode_update.
 */
ckv_status ckv_kpool_compress(uint8_t* kv_cache, int64_t num_pages, int32_t page_size,
                              const uint16_t* slot_k, const uint16_t* slot_score, const float* ape,
                              const int64_t* loc, const uint8_t* write_mask, int32_t write_cache,
                              uint8_t* out_fp8, float* out_scale, int64_t n_pools, int32_t P,
                              int32_t D, int32_t round_scale, float* tap_x, uint16_t* tap_xb,
                              uint16_t* tap_yb, int32_t use_pdl, int32_t* err_word, void* stream);

/*
 * Seed the pooled tail ring from a prefill batch (vLLM kpool_compress page,
 * _kpool_tail_seed_kernel and kpool_seed_tail_cache).  Token i with tail slot
 * t = tslot[i] >= 0 is copied to ring[t / P][{key, score}][t % P] iff the
 * token P places ahead (i + P) is past the batch, has a negative tail slot,
 * or lies in another tail block -- i.e. the token is among its request's
 * last P tokens.
 * key, score  device bf16 [n_tokens][D] contiguous; tslot device int32 [n_tokens].
 * tail_ring   device bf16 [num_tail_blocks][2][P][D].  P in {1,2,4,8,16}; D == 128.
 */
ckv_status ckv_kpool_seed_tail(uint16_t* tail_ring, int64_t num_tail_blocks, const uint16_t* key,
                               const uint16_t* score, const int32_t* tslot, int64_t n_tokens,
                               int32_t P, int32_t D, int32_t* err_word, void* stream);

/*
 * Pool -> token index expansion with the tail appended (vLLM kpool_compress
 * page, expand_pools_and_append_tail: the identity path of
 * expand_pools_to_tokens followed by append_tail_to_topk).  For row r with
 * s = seq_lens[r] and G = n_groups, out[r] has G*P + P - 1 int32 columns:
 *   column g*P + o  = pool_ids[r][g] * P + o, or -1 when pool_ids[r][g] < 0;
 *   column G*P + i  = (s / P) * P + i when i < s % P (the tokens of the
 *                     unfinished trailing pool), else -1.
 * pool_ids  device int32, row r at r * pool_ids_stride (>= n_groups) elements;
 *           n_groups <= 2048 (a top-k of up to 2048 * P tokens).
 * seq_lens  device int64 [rows], >= 0.     out  device int32 [rows][G*P + P - 1].
 * P         1..1024 (P = 1 has no tail columns).
 */
ckv_status ckv_expand_pools_and_append_tail(const int32_t* pool_ids, int64_t pool_ids_stride,
                                           const int64_t* seq_lens, int32_t rows, int32_t n_groups,
                                           int32_t P, int32_t* out, int32_t use_pdl, void* stream);

/*
 * Online c128 decode (sglang c128_online.cuh page, flash_c128_online_decode
 * and run_decode).  For request b: the token sits at chunk position
 * p = (seq_lens[b] - 1) % 128 with logit z = score + ape[p].
 *   p == 0:   state := (z, 1, kv_in)
 *   p  > 0:   merge into the state of slot indices[b]:
 *             M = max(m, z), s' = s*e^(m-M) + e^(z-M),
 *             kv' = (kv*s*e^(m-M) + kv_in*e^(z-M)) / s'
 *   p == 127: out[b] := kv' and the slot is left unchanged; otherwise the
 *             new (max, sum, kv) is stored in slot indices[b].
 * state       device fp32 [num_slots][3][D] laid out max | sum | kv.
 * input       device [B][2D] laid out kv | score; fp32 (CKV_F32) or bf16 (CKV_BF16).
 * out         device fp32 [B][D]; only rows of chunk-closing requests are written.
 * ape         device fp32 [128][D].   indices, seq_lens: device int32 [B].
 * D           128, 256 or 512.   Pointers 16-byte aligned.
 * use_pdl     nonzero: launch as a programmatic dependent launch (the kernel
 *             waits for the preceding grid before touching memory).
 */
ckv_status ckv_c128_online_decode(float* state, int64_t num_slots, const void* input,
                                  ckv_dtype in_dtype, float* out, const float* ape,
                                  const int32_t* indices, const int32_t* seq_lens, int32_t B,
                                  int32_t D, int32_t use_pdl, int32_t* err_word, void* stream);

/*
 * Online c128 prefill (sglang c128_online.cuh page, flash_c128_online_prefill,
 * c128_prefill_forward and run_prefill).  Two stream-ordered launches:
 *   1. compress pass over compress_plan[0..num_compress): per segment and
 *      channel, softmax over the segment's tokens (bias ape[chunk position]),
 *      merged with the partial state of slot load_indices[batch_id] when the
 *      segment does not start at chunk position 0; the result is written to
 *      out[ragged_id].  The state buffer is only read.
 *   2. write pass over write_plan[0..num_write): the same reduction, whose
 *      (max, sum, kv) is stored into slot indices[batch_id].
 * The second pass touches the state only after the first pass has completed,
 * so a slot read in pass 1 may be overwritten in pass 2.  With use_pdl the
 * second pass may start reading its plan, indices and input tokens while the
 * first pass still runs (nothing it reads except the state is written by the
 * first pass); without it the two launches are plainly stream ordered.
 * state          device fp32 [num_slots][3][D].
 * input          device [num_tokens][2D] (kv | score), fp32 or bf16.
 * out            device fp32 [num_tokens][D]; only compress rows are written.
 * ape            device fp32 [128][D].
 * indices        device int32 [B]; load_indices device int32 [B] or NULL (= indices).
 * compress_plan, write_plan
 *                device arrays of ckv_plan_entry (16-byte aligned), e.g. from
 *                ckv_plan_online_prefill; sentinel entries are skipped.
 * D              128, 256 or 512.   use_pdl as for decode.
 */
ckv_status ckv_c128_online_prefill(float* state, int64_t num_slots, const void* input,
                                   ckv_dtype in_dtype, int64_t num_tokens, float* out,
                                   const float* ape, const int32_t* indices,
                                   const int32_t* load_indices, int32_t B,
                                   const ckv_plan_entry* compress_plan, uint32_t num_compress,
                                   const ckv_plan_entry* write_plan, uint32_t num_write, int32_t D,
                                   int32_t use_pdl, int32_t* err_word, void* stream);

/*
 * Kernel choice for the compress pass of ckv_c128_online_prefill (process-wide).
 *   0 = automatic (default): the TMA-pipelined persistent kernel when there
 *       are at least 1024 compress segments, otherwise the one-CTA-per-segment
 *       kernel;
 *   1 = always the one-CTA-per-segment kernel;
 *   2 = always the TMA-pipelined kernel (when the device supports it).
 * Both compute the same function.  Returns the previous setting, or -1 (and
 * changes nothing) for an unknown value.
 */
int32_t ckv_c128_prefill_set_variant(int32_t variant);

/*
 * Kernel choice for ckv_kpool_compress (process-wide).
 *   0 = automatic (default): the persistent bulk-copy pipeline for at least
 *       65536 pools, otherwise one warp per pool;
 *   1 = always one warp per pool;  2 = always the bulk-copy pipeline.
 * Both compute the same function.  Returns the previous setting, or -1 (and
 * changes nothing) for an unknown value.
 */
int32_t ckv_kpool_compress_set_variant(int32_t variant);

/*
 * Host planner for the online c128 prefill (sglang c128_online.cuh page,
 * plan_online_prefill_host).  Request i covers global positions
 * [seq_lens[i] - extend_lens[i], seq_lens[i]) and ragged rows that follow the
 * rows of requests 0..i-1.  The range is split at multiples of 128; a
 * segment ending at chunk position 127 is appended to compress_plan, the
 * trailing partial segment (at most one per request) to write_plan.
 * seq_lens, extend_lens  host int64 [B]; 0 < extend_lens[i] <= seq_lens[i] < 2^32.
 * num_tokens             must equal sum(extend_lens); it is also the capacity
 *                        (rows) of each plan array.
 * compress_plan, write_plan host (or pinned) arrays of num_tokens entries.
 * pad_for_graph          nonzero: fill both arrays to num_tokens rows with
 *                        sentinels and report num_tokens for both counts, so
 *                        a captured CUDA graph always sees the same grid.
 * num_compress, num_write host outputs.
 * Returns CKV_ERR_PLAN (and writes no counts) on invalid lengths.
 */
ckv_status ckv_plan_online_prefill(const int64_t* seq_lens, const int64_t* extend_lens, uint32_t B,
                                   uint32_t num_tokens, ckv_plan_entry* compress_plan,
                                   ckv_plan_entry* write_plan, int32_t pad_for_graph,
                                   uint32_t* num_compress, uint32_t* num_write);

/*
 * The c128 calls with an FP8 output stage: every compressed row the call
 * emits (decode: the rows of chunk-closing requests; prefill: the compress
 * rows) is also stored into a paged FP8 cache, the way the pooled path stores
 * its rows -- the combination of the sglang c128_online.cuh page's
 * compressed rows with the quantisation stage of the vLLM kpool_compress
 * page (_kpool_softmax_rotate_write_cache_kernel).  Neither page shows this
 * combination; the readings taken:
 *   - the row's D channels are D/128 blocks of 128, and each block is treated
 *     exactly like one pooled vector: fp32 -> bf16 (round to nearest even) ->
 *     Hadamard-128 (the pooled path's rotation) -> bf16 -> absmax FP8-e4m3 with
 *     its own fp32 scale (round_scale as for the pooled calls);
 *   - kv_cache  device uint8 [num_pages][page_size][D + 4*(D/128)]: per page,
 *     page_size rows of D FP8 bytes (block j at bytes 128j..128j+127), then
 *     page_size*(D/128) fp32 scales (row r, block j at r*(D/128) + j); with
 *     D = 128 this is the pooled cache layout.
 * cache_loc   device int64: decode [B], the cache row of request b when its
 *             chunk closes; prefill [num_tokens], read at the ragged row of
 *             each compress segment.  A location outside
 *             [0, num_pages*page_size) sets CKV_DEVERR_CACHE_LOC and is skipped.
 * out         may be NULL here (only the FP8 rows are produced); otherwise as
 *             for ckv_c128_online_decode / ckv_c128_online_prefill.
 * All other arguments and the state update are those of the plain calls.
 */
ckv_status ckv_c128_online_decode_fp8(float* state, int64_t num_slots, const void* input,
                                      ckv_dtype in_dtype, float* out, const float* ape,
                                      const int32_t* indices, const int32_t* seq_lens, int32_t B,
                                      int32_t D, uint8_t* kv_cache, int64_t num_pages,
                                      int32_t page_size, const int64_t* cache_loc,
                                      int32_t round_scale, int32_t use_pdl, int32_t* err_word,
                                      void* stream);
ckv_status ckv_c128_online_prefill_fp8(float* state, int64_t num_slots, const void* input,
                                       ckv_dtype in_dtype, int64_t num_tokens, float* out,
                                       const float* ape, const int32_t* indices,
                                       const int32_t* load_indices, int32_t B,
                                       const ckv_plan_entry* compress_plan, uint32_t num_compress,
                                       const ckv_plan_entry* write_plan, uint32_t num_write,
                                       int32_t D, uint8_t* kv_cache, int64_t num_pages,
                                       int32_t page_size, const int64_t* cache_loc,
                                       int32_t round_scale, int32_t use_pdl, int32_t* err_word,
                                       void* stream);

/*
 * Device-side planner: the same plans as ckv_plan_online_prefill (sglang
 * c128_online.cuh page, plan_online_prefill_host), computed by a CUDA kernel
 * on `stream`, so that planning and the prefill can be enqueued -- or
 * captured in a CUDA graph -- without a host round trip.
 * seq_lens, extend_lens  device int64 [B]; B <= 8192.
 * compress_plan, write_plan device arrays of num_tokens entries (16-byte aligned).
 * counts                 device uint32 [2]: receives (num_compress, num_write),
 *                        both num_tokens with pad_for_graph.
 * Invalid lengths (extend <= 0, extend > seq, seq >= 2^32, sum != num_tokens)
 * set CKV_DEVERR_PLAN in err_word and write counts (0, 0).
 */
ckv_status ckv_plan_online_prefill_device(const int64_t* seq_lens, const int64_t* extend_lens,
                                          uint32_t B, uint32_t num_tokens,
                                          ckv_plan_entry* compress_plan, ckv_plan_entry* write_plan,
                                          int32_t pad_for_graph, uint32_t* counts, int32_t use_pdl,
                                          int32_t* err_word, void* stream);

/*
 * ckv_c128_online_prefill with the segment counts read on the device from
 * `counts` (device uint32 [2] = num_compress, num_write, e.g. written by
 * ckv_plan_online_prefill_device) instead of passed by the host.  The grids
 * are sized for the largest possible counts (num_tokens/128 + B compress and B
 * write segments); the kernels clamp the device counts to those bounds.  All
 * other arguments as for ckv_c128_online_prefill.
 */
ckv_status ckv_c128_online_prefill_counted(float* state, int64_t num_slots, const void* input,
                                           ckv_dtype in_dtype, int64_t num_tokens, float* out,
                                           const float* ape, const int32_t* indices,
                                           const int32_t* load_indices, int32_t B,
                                           const ckv_plan_entry* compress_plan,
                                           const ckv_plan_entry* write_plan, const uint32_t* counts,
                                           int32_t D, int32_t use_pdl, int32_t* err_word,
                                           void* stream);

/*
 * Debug check of the caller contract (no counterpart in the sources, which
 * state the contract and leave it unchecked).  Within one call the kernels
 * above need distinct state slots (`indices` of the c128 calls), distinct
 * cache locations (`slot_mapping`, `loc` of the pooled calls) and a tail
 * block per request that no other request uses; a repeat is a data race that
 * no kernel detects.  This call checks one such list: it ORs
 * CKV_DEVERR_DISTINCT into *err_word when one of the first n ids repeats or
 * is >= range.  Negative ids (padding) are ignored.  For tail blocks, pass one
 * block id per request.
 *   ids        device, n int32 (id_bytes = 4) or int64 (id_bytes = 8)
 *   range      ids are expected in [0, range); 1 <= range <= 2^40
 *   scratch    device uint32 [scratch_words], scratch_words >= ceil(range/32),
 *              owned by the caller; cleared and then used as a bitmap (one bit
 *              per id), so its contents on return are not meaningful
 *   err_word   device int32, required
 * Enqueues two kernels (clear, mark) on `stream`.  Calls that share `scratch`
 * and overlap on the GPU race.  n == 0 clears the scratch and checks nothing.
 */
ckv_status ckv_check_distinct(const void* ids, int32_t id_bytes, int64_t n, int64_t range,
                              uint32_t* scratch, int64_t scratch_words, int32_t* err_word,
                              void* stream);

/*
 * ckv_check_distinct without a scratch argument, for callers that cannot
 * allocate device memory: e.g. a serving engine that has reserved nearly all
 * HBM for its paged KV cache and hands out no other buffers, or a loop that
 * must not call cudaMalloc because it may synchronise the device.  No source
 * page describes this check (a debugging aid).  The bitmap is a static device array of
 * CKV_NOALLOC_MAX_RANGE bits (256 KB) inside the library, held by every GPU
 * that loads it until the process exits; the library allocates nothing.
 *   ids, id_bytes, n, err_word, stream  as for ckv_check_distinct
 *   range      1 <= range <= CKV_NOALLOC_MAX_RANGE; a larger range returns
 *              CKV_ERR_SHAPE and launches nothing
 * The first call on each device looks up the array's device address (with
 * that device current) and keeps it; make that first call before any stream
 * capture.  The kept address belongs to the device's context of that moment:
 * do not reset the device (cudaDeviceReset) after the first call in a process
 * that calls this again.  Every call uses the same array: it is cleared at the
 * start of each call, and calls that overlap on the GPU (other streams, other
 * threads) race.
 */
#define CKV_NOALLOC_MAX_RANGE (1 << 21)
ckv_status ckv_check_distinct_noalloc(const void* ids, int32_t id_bytes, int64_t n, int64_t range,
                                      int32_t* err_word, void* stream);

/*
 * ckv_c128_online_prefill_counted with the FP8 output stage of
 * ckv_c128_online_prefill_fp8 (same readings, cache layout and cache_loc,
 * read at the ragged row of each compress segment; out may be NULL).
 */
ckv_status ckv_c128_online_prefill_counted_fp8(float* state, int64_t num_slots, const void* input,
                                               ckv_dtype in_dtype, int64_t num_tokens, float* out,
                                               const float* ape, const int32_t* indices,
                                               const int32_t* load_indices, int32_t B,
                                               const ckv_plan_entry* compress_plan,
                                               const ckv_plan_entry* write_plan,
                                               const uint32_t* counts, int32_t D, uint8_t* kv_cache,
                                               int64_t num_pages, int32_t page_size,
                                               const int64_t* cache_loc, int32_t round_scale,
                                               int32_t use_pdl, int32_t* err_word, void* stream);

/*
 * Latency floor of a decode-sized launch: a measurement aid with no
 * counterpart in the sources.  Launches n_warps warps, warps_per_cta to a CTA
 * (the pooled decode update's launch shape is one CTA of two warps per
 * request), each of which first waits for the preceding grid when use_pdl is set
 * (programmatic dependent launch), then does only dependent memory traffic:
 *   hops == 0  nothing (the cost of launching and completing the grid);
 *   hops == 1  loads idx[w] and stores it to the first 4 bytes of row w of out
 *              (one global round trip);
 *   hops == 2  loads idx[w], then row idx[w] of rows, and stores it as row w
 *              of out (two dependent round trips, as when a closing pool's
 *              index words name the ring rows it reads).
 *   hops == 3  one round trip with the pooled decode's first-hop loads: each
 *              thread loads 12 words of idx[b0 .. b0 + 15] (b0 = w rounded
 *              down to a multiple of 4, at most n_warps - 16) and 8 four-byte
 *              words of rows 256 bytes apart, starting at word
 *              (8w mod (64 num_rows - 512)) + lane; lane 0 stores the
 *              exclusive or of the 20 words it loaded (idx[w] among them) to
 *              the first 4 bytes of row w of out.  Needs n_warps >= 16 and
 *              num_rows >= 9.
 *   hops == 4  the pooled decode's memory pattern without its arithmetic:
 *              the index loads of hops == 3 and 8 row words per thread from
 *              the warp pair's own 2 KB (starting at word ((w / 2) 512 mod
 *              (64 num_rows - 512)) + 32 (w mod 2) + lane, 256 bytes apart:
 *              8 rows, a half-row for each warp, as a request's 4 key and 4
 *              score rows); then warps whose pair index (w / 2) is a multiple
 *              of 4 (a request whose pool closes) load, if 0 <= idx[w] <
 *              num_rows, 30 words per thread from the 8 KB block min(idx[w] /
 *              32, num_rows / 32 - 1) of rows (32 rows each): rows 0..14 and
 *              16..30, at word 32 (w mod 2) + lane of each (as a closing
 *              pool's 15 key and 15 score ring rows); then each thread stores
 *              its 8 first-hop row words to bytes [1024 w, 1024 w + 1024) of
 *              out (word q of lane l at word 256 w + 32 q + l), as the ring
 *              stashes of a request's tokens; lane 0 finally stores the
 *              exclusive or of every word it loaded to the first 4 bytes of
 *              warp w's kilobyte.  Needs n_warps >= 16 and num_rows >= 64.
 *   idx        device int32 [n_warps] (hops >= 1); an index outside
 *              [0, num_rows) makes that warp skip its row (hops == 2) or its
 *              second hop (hops == 4)
 *   rows       device [num_rows][256 bytes], 8-byte aligned (hops >= 2)
 *   out        device [n_warps][256 bytes] (hops 1..3) or [4 n_warps][256
 *              bytes] (hops == 4), 8-byte aligned
 * Sizes outside hops 0..4, 1 <= n_warps <= 2^30, 1 <= warps_per_cta <= 32
 * (and the hops == 3 and 4 minimums) return CKV_ERR_SHAPE and launch
 * nothing.
 */
ckv_status ckv_latency_probe(int32_t hops, const int32_t* idx, const void* rows, int64_t num_rows, void* out,
                             int32_t n_warps, int32_t warps_per_cta, int32_t use_pdl, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CKV_H_ */
