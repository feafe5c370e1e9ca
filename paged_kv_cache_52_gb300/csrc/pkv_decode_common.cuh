// Shared by the bf16 and FP8 decode kernels: launch parameters and the
// clamping of a sequence's length to what its block table and the split plan
// cover (both kernels and the merge must agree on it).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace pkv {

constexpr int kBlockTokens = 16;  // tokens per KV page

// Blocks of a sequence the kernels attend over, after clamping to what the
// block table and the plan cover.  Both kernels use this so they agree.
__device__ __forceinline__ int effective_blocks(int len, int max_blocks_per_seq, int num_parts,
                                                int partition_blocks, bool* bad) {
  *bad = false;
  if (len < 0) {
    len = 0;
    *bad = true;
  }
  int nblk = (len + kBlockTokens - 1) / kBlockTokens;
  if (nblk > max_blocks_per_seq) {
    nblk = max_blocks_per_seq;
    *bad = true;
  }
  const int covered = num_parts * partition_blocks;
  if (nblk > covered) {
    nblk = covered;
    *bad = true;
  }
  return nblk;
}

__device__ __forceinline__ int effective_len(int len, int nblk) {
  len = len < 0 ? 0 : len;
  return len < nblk * kBlockTokens ? len : nblk * kBlockTokens;
}

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
};


cudaError_t launch_decode_merge(const DecodeParams& prm, int num_seqs, int d_head,
                                cudaStream_t stream);

}  // namespace pkv
