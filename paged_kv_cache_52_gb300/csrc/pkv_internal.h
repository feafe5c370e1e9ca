// Host-side launch entry points of each kernel translation unit, called by
// the C ABI layer (pkv_api.cu).  Arguments are validated before these run.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace pkv {

// Every kernel unit keeps its own device error word (an OR of the
// PKV_DEVERR_* bits its kernels raised); <unit>_error_word gives its device
// address on the current device.
cudaError_t append_error_word(unsigned** word);
cudaError_t decode_error_word(unsigned** word);
cudaError_t decode_fp8_error_word(unsigned** word);
cudaError_t prefill_error_word(unsigned** word);
cudaError_t verify_error_word(unsigned** word);
cudaError_t probe_error_word(unsigned** word);
cudaError_t mixed_decode_error_word(unsigned** word);
cudaError_t mixed_prefill_error_word(unsigned** word);
cudaError_t decode_flat_error_word(unsigned** word);

// ---- kv_append.cu
// reject (optional): a device flag set by launch_slot_duplicates; when it is
// nonzero the append writes nothing.
cudaError_t launch_kv_append(const void* k, int64_t k_stride, const void* v, int64_t v_stride,
                             const int64_t* slot_mapping, int64_t num_tokens, void* k_cache,
                             void* v_cache, int64_t num_slots, int row_elems,
                             cudaStream_t stream, int num_sms, const int* reject = nullptr,
                             bool trigger_dependents = false);
// Marks every in-pool slot in `bitmap` (num_slots bits, zeroed by the
// caller) and sets *reject when a slot repeats.
cudaError_t launch_slot_duplicates(const int64_t* slot_mapping, int64_t num_tokens,
                                   int64_t num_slots, unsigned* bitmap, int* reject,
                                   cudaStream_t stream, int num_sms);
unsigned read_append_error(bool clear);
// FP8 (e4m3) pools: row_elems must be a multiple of 16.
cudaError_t launch_kv_append_fp8(const void* k, int64_t k_stride, const void* v, int64_t v_stride,
                                 const int64_t* slot_mapping, int64_t num_tokens, void* k_cache,
                                 void* v_cache, int64_t num_slots, int row_elems, float k_inv,
                                 float v_inv, cudaStream_t stream, int num_sms);
// FP8 pages of each sequence's context -> bf16 scratch pool + scratch table
// (page_codes = 16 * kv_heads * d_head, a multiple of 16).  seq_order
// (optional, [num_seqs]): the sequences by context length, longest first,
// ties by index -- the prefill's dispatch order.
cudaError_t launch_widen_fp8_pages(const void* k8, const void* v8, const int32_t* tables,
                                   const int32_t* lens, int num_seqs, int max_blocks,
                                   int num_blocks, int64_t page_codes, void* kdst, void* vdst,
                                   int32_t* table_out, bool v_f16, int32_t* seq_order,
                                   cudaStream_t stream, int num_sms);
// bf16 V pages of each sequence's context -> f16 scratch pool + scratch table
// (page_elems = 16 * kv_heads * d_head, a multiple of 8); seq_order as above.
cudaError_t launch_v_pages_to_f16(const void* v, const int32_t* tables, const int32_t* lens,
                                  int num_seqs, int max_blocks, int num_blocks, int64_t page_elems,
                                  void* vdst, int32_t* table_out, int32_t* seq_order,
                                  cudaStream_t stream, int num_sms);
// ---- wait_probe.cu
// Bounded-wait probe: one thread waits on an mbarrier phase that never
// completes, with `polls` (1 .. kWaitPollLimit) as the poll limit; the wait
// gives up and the timeout bit is recorded.  cycles (optional, device): the
// clock64 cycles the wait took.
cudaError_t launch_wait_timeout_probe(uint32_t polls, unsigned long long* cycles,
                                      cudaStream_t stream);
unsigned read_probe_error(bool clear);
uint32_t wait_poll_limit();

// Copy-on-write block copies: block_bytes a multiple of 16.
cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs,
                               int num_blocks, int64_t block_bytes, cudaStream_t stream,
                               int num_sms);

// ---- paged_decode.cu
struct DecodeArgs {
  const void* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* out;
  float* part_o;    // [S][Hq][num_parts][d] (num_parts > 1 only)
  float* part_lse;  // [S][Hq][num_parts]
  int num_seqs, q_heads, kv_heads, d_head, num_blocks;
  int max_blocks_per_seq;
  int partition_blocks, num_parts;
  float scale_log2;  // scale * log2(e)
  float out_scale;   // FP8 pools: the V dequantization scale (1 for bf16)
  // cascade (shared prefix): skip the first blocks, always write partials,
  // merge in one extra normalised partial per row
  int first_block = 0;
  int force_partials = 0;
  const float* extra_o = nullptr;
  const float* extra_lse = nullptr;
  // prefix groups: per-sequence first block (null: first_block for all)
  const int32_t* seq_first_block = nullptr;
  // the split kernel lets the next grid start while it runs (that grid must
  // wait for it before finishing); skip_merge: launch the split kernel only
  // (launch_paged_decode_merge_only launches the merge)
  bool early_trigger = false;
  bool skip_merge = false;
  // the split kernel starts beside the append launched just before it and
  // waits for that append only before loading a sequence's last page (the
  // one holding its appended token); the decode-step entry point sets it
  bool wait_late = false;
  const int64_t* step_slots = nullptr;  // with wait_late: the append's slot mapping
  bool out_bf16 = false;  // out is bf16 (rounded to nearest even), not float32
  // length-balanced work list (bf16 decode): list_items CTAs (an upper bound
  // on the runs), partials at part_o / part_lse indexed by run * G + head,
  // and the per-sequence first runs at list_base ([num_seqs + 1] int32)
  bool list = false;
  int32_t* list_base = nullptr;
  int list_target = 0, list_min_run = 0, list_max_blocks = 0, list_items = 0;
  int list_max_ctas = 0;  // > 0: at most this many CTAs, each looping over runs
  // flat split (bf16 decode): flat_ctas CTAs (one per SM) whose warps each
  // stream one contiguous range of the pages of all pairs laid end to end;
  // partials at part_o / part_lse indexed by (pair + warp) * G + head, the
  // page prefix sums at flat_pre ([num_seqs + 1] int32), at most
  // flat_max_blocks pages per sequence
  bool flat = false;
  int32_t* flat_pre = nullptr;
  int flat_ctas = 0, flat_max_blocks = 0;
  bool fp8 = false;  // flat split over FP8 (e4m3) pools, out_scale = v_scale
};

// Multi-query decode (speculative verification): q_len query tokens per
// sequence, rows (seq * q_len + t) * q_heads + head of q and out; group *
// q_len <= verify_max_rows().  Uses the decode plan and workspace layout with
// num_seqs * q_len rows per head.
int verify_max_rows();
cudaError_t launch_paged_verify(const DecodeArgs& a, int q_len, const CUtensorMap* tmap_k,
                                const CUtensorMap* tmap_v, cudaStream_t stream);
unsigned read_verify_error(bool clear);

// Prefix groups: for each sequence, the first block of its own pages (the
// group's prefix length in blocks, or 0 when it has no group, its group's
// prefix is out of range, longer than its context, or its first ids differ
// from the group leader's -- those set PKV_DEVERR_PREFIX_MISMATCH), and for
// each group the prefix length in tokens (0 for an invalid one).
// group_start null: one group of every sequence with uniform_prefix_blocks.
cudaError_t launch_prefix_groups_setup(const int32_t* group_start,
                                       const int32_t* group_prefix_blocks, int num_groups,
                                       int uniform_prefix_blocks, int num_seqs,
                                       const int32_t* block_tables, int max_blocks_per_seq,
                                       const int32_t* context_lens, int max_prefix_blocks,
                                       int32_t* seq_first_block, int32_t* group_ctx,
                                       cudaStream_t stream);

// Number of K/V stages and warps the decode kernel uses (for the plan).
int decode_warps_per_cta();
int decode_max_partition_blocks();
int decode_list_max_seqs();

cudaError_t launch_paged_decode(const DecodeArgs& a, const CUtensorMap* tmap_k,
                                const CUtensorMap* tmap_v, cudaStream_t stream);
cudaError_t launch_paged_decode_merge_only(const DecodeArgs& a, cudaStream_t stream);
unsigned read_decode_error(bool clear);

// ---- paged_decode_flat.cu (the flat split of the bf16 decode, and its merge)
// warps of a flat CTA over bf16 or FP8 pools (0: d_head not supported)
int decode_flat_warps(int d_head, bool fp8 = false);
int decode_flat_max_seqs();
// the kernel, then (unless skip_merge) its merge; with seq_first_block /
// first_block and extra_o / extra_lse as in the cascade decode
cudaError_t launch_paged_decode_flat(const DecodeArgs& a, const CUtensorMap* tmap_k,
                                     const CUtensorMap* tmap_v, cudaStream_t stream);
cudaError_t launch_paged_decode_flat_merge(const DecodeArgs& a, cudaStream_t stream);
unsigned read_decode_flat_error(bool clear);

// ---- paged_decode_fp8.cu (e4m3 pools, d_head 128)
cudaError_t launch_paged_decode_fp8(const DecodeArgs& a, const CUtensorMap* tmap_k,
                                    const CUtensorMap* tmap_v, cudaStream_t stream);
unsigned read_decode_fp8_error(bool clear);

// ---- paged_prefill.cu
struct PrefillArgs {
  const int32_t* q_start;       // null: one sequence owning all total_q rows
  const int32_t* block_tables;
  const int32_t* context_lens;  // null: context_len below
  float* out;
  float* lse = nullptr;         // optional per-row log2-sum-exp
  float out_scale = 1.f;        // multiplies the output (FP8 pools: v_scale)
  // V from its own (f16) pool through its own table, P as one f16 operand
  bool f16_pv = false;
  const int32_t* v_block_tables = nullptr;  // null: block_tables
  int v_num_blocks = 0;
  int context_len = 0;
  int num_seqs, total_q, max_q_len, q_heads, kv_heads, d_head, num_blocks;
  int max_blocks_per_seq;
  int causal;
  float scale_log2;
  // > 0: persistent launch of at most max_ctas CTAs taking query tiles from
  // work_counter (one int of device memory, zeroed by the launch)
  int max_ctas = 0;
  int* work_counter = nullptr;
  bool out_bf16 = false;  // out is bf16 (rounded to nearest even), not float32
  // optional [num_seqs]: sequences in dispatch order (longest context first);
  // null: index order
  const int32_t* seq_order = nullptr;
  // optional [num_seqs]: the block_tables row of each sequence (prefix
  // groups: the leader's row); null: its own row
  const int32_t* table_rows = nullptr;
  bool allow_empty = false;  // a context of 0 is skipped without a flag
  // the grid starts without waiting for the kernel before it (which let it
  // start early and wrote nothing it reads) and waits for that kernel only
  // before it finishes, so the next kernel sees both complete
  bool defer_wait = false;
};

// Query rows (tokens x heads of a GQA group) per prefill tile.
int prefill_rows_per_tile();

// tmap_o (optional): the float32 output as d_head x q_heads x total_q, box
// 32 columns x G heads x 32/G tokens, 128-byte swizzled (encode_out_map);
// with it whole warps' rows are written by TMA stores
cudaError_t launch_paged_prefill(const PrefillArgs& a, const CUtensorMap* tmap_q,
                                 const CUtensorMap* tmap_k, const CUtensorMap* tmap_v,
                                 cudaStream_t stream, const CUtensorMap* tmap_o = nullptr);
unsigned read_prefill_error(bool clear);

// ---- mixed_step.cu
// The continuous-batching step's attention in one persistent launch of
// `ctas` CTAs: pa describes the chunked prefill (f16 P V path: V through
// pa.v_block_tables into the f16 scratch pool, which tmap_v16 maps), da the
// bf16 decode as a length-balanced list (da.list_* set, partials in
// da.part_o / part_lse).  Launches the decode plan, the fused kernel and the
// list merge.  counter: one int of device memory.
// prefix (optional): the decode prefix groups' pass (bf16 V from the pool,
// queries through tmap_qd); da then carries seq_first_block and the extra
// partial's buffers.  tmap_o (optional): the prefill output map of
// launch_paged_prefill, for TMA stores of the prefill items' rows.
cudaError_t launch_mixed_step(const PrefillArgs& pa, const DecodeArgs& da, int* counter,
                              int ctas, int prefill_span_permille, const CUtensorMap* tmap_q,
                              const CUtensorMap* tmap_k, const CUtensorMap* tmap_v16,
                              const CUtensorMap* tmap_v, cudaStream_t stream,
                              const PrefillArgs* prefix = nullptr,
                              const CUtensorMap* tmap_qd = nullptr,
                              const CUtensorMap* tmap_o = nullptr);
unsigned read_mixed_error(bool clear);

}  // namespace pkv
