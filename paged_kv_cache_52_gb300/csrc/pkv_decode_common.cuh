// Shared by the bf16 and FP8 decode kernels: launch parameters and the
// clamping of a sequence's length to what its block table and the split plan
// cover (both kernels and the merge must agree on it).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace pkv {

constexpr int kBlockTokens = 16;  // tokens per KV page

struct DecodeParams {
  const __nv_bfloat16* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* out;
  float* part_o;
  float* part_lse;
  int q_heads, kv_heads, num_blocks, max_blocks_per_seq, partition_blocks, num_parts;
  float scale_log2;  // softmax scale (times the K dequantization scale) * log2(e)
  float out_scale;   // multiplies the normalised output (the V dequantization scale)
  // Cascade (shared-prefix) mode: attend only blocks [first_block, ...), always
  // write partials, and let the merge fold in one extra partial per row.
  int first_block;
  int force_partials;
  const float* extra_o;    // [S][q_heads][d] normalised output of the extra part, or null
  const float* extra_lse;  // [S][q_heads] its log2-sum-exp
  // nonzero: out holds bf16 (the fp32 result rounded to nearest even)
  int out_bf16 = 0;
  // prefix groups: sequence s attends blocks [seq_first_block[s], ...) and
  // merges the extra partial only when that is nonzero (null: first_block)
  const int32_t* seq_first_block = nullptr;
  // nonzero: the split kernel lets the next grid (a prefix pass that waits
  // for this grid only at its end) start while it runs
  int early_trigger = 0;
  // nonzero: the grid before this one is the step's append, which let this
  // grid start early; only the loads of a sequence's last page wait for it
  // (that page holds the appended token; the append writes nothing else the
  // decode reads when every slot is its sequence's position context_len - 1)
  int wait_late = 0;
  const int64_t* step_slots = nullptr;  // the append's slot mapping (wait_late), for a check
};

// First block a sequence's own pages start at (0: no shared prefix).
__device__ __forceinline__ int first_block_of(const DecodeParams& p, int seq) {
  return p.seq_first_block ? p.seq_first_block[seq] : p.first_block;
}

// Whether the row's sequence merges the extra (shared-prefix) partial.
__device__ __forceinline__ bool has_extra(const DecodeParams& p, int seq) {
  return p.extra_o != nullptr && first_block_of(p, seq) > 0;
}

// Store element i of the final output in the caller's precision.
__device__ __forceinline__ void store_out(const DecodeParams& p, size_t i, float v) {
  if (p.out_bf16)
    reinterpret_cast<__nv_bfloat16*>(p.out)[i] = __float2bfloat16_rn(v);
  else
    p.out[i] = v;
}

// The blocks of a sequence the kernels attend over: [first, first + count),
// after clamping to what the block table and the split plan cover, and the
// context length clamped to match.  The split kernels and the merge use this
// so they agree.
struct SeqSpan {
  int len;    // attended positions end here
  int first;  // first block attended
  int count;  // blocks attended
  bool bad;   // the context length had to be clamped
};

__device__ __forceinline__ SeqSpan seq_span(int raw_len, const DecodeParams& p, int seq) {
  SeqSpan sp;
  sp.bad = false;
  int len = raw_len;
  if (len < 0) {
    len = 0;
    sp.bad = true;
  }
  int nblk = (len + kBlockTokens - 1) / kBlockTokens;
  if (nblk > p.max_blocks_per_seq) {
    nblk = p.max_blocks_per_seq;
    sp.bad = true;
  }
  sp.first = first_block_of(p, seq);
  if (sp.first > 0 && len < sp.first * kBlockTokens) sp.bad = true;  // shorter than the prefix
  sp.count = nblk > sp.first ? nblk - sp.first : 0;
  const int covered = p.num_parts * p.partition_blocks;
  if (sp.count > covered) {
    sp.count = covered;
    sp.bad = true;
  }
  const int end = (sp.first + sp.count) * kBlockTokens;
  sp.len = len < end ? len : end;
  return sp;
}

// Partitions a sequence's span splits into (0 with an empty span in cascade
// mode, where the extra partial carries the whole result).
__device__ __forceinline__ int span_parts(const SeqSpan& sp, const DecodeParams& p) {
  if (sp.count == 0) return p.force_partials ? 0 : 1;
  return (sp.count + p.partition_blocks - 1) / p.partition_blocks;
}

cudaError_t launch_decode_merge(const DecodeParams& prm, int num_seqs, int d_head,
                                cudaStream_t stream);

// The length-balanced list of runs (see list_plan).
struct DecodeListParams {
  int32_t* seq_item_base;  // [num_seqs + 1]: first run of each sequence, then the run count
  int num_seqs;            // <= kListMaxSeqs
  int target_items;        // runs aimed at
  int min_run;             // pages
  int max_blocks;          // page bound per sequence (block table and host max_context_len)
};

// Pages of a sequence in the list plan: its context clamped to max_blocks.
__device__ __forceinline__ int list_pages(int len, int max_blocks) {
  int n = len <= 0 ? 0 : (len + kBlockTokens - 1) / kBlockTokens;
  return n < max_blocks ? n : max_blocks;
}

// The sequence's own pages in the list plan (after its shared prefix), and
// the first of them.
__device__ __forceinline__ int list_own_pages(const DecodeParams& p, const DecodeListParams& lp,
                                              int seq, int* first) {
  const int f = first_block_of(p, seq);
  const int n = list_pages(p.context_lens[seq], lp.max_blocks) - f;
  *first = f;
  return n > 0 ? n : 0;
}

// The merge of a list decode's runs (after the kernel that wrote them).
cudaError_t launch_decode_list_merge(const DecodeParams& prm, const DecodeListParams& lp,
                                     int d_head, cudaStream_t stream);

}  // namespace pkv
