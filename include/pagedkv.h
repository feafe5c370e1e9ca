/*
 * pagedkv.h -- C ABI of the GB300 (sm_103a) paged-KV attention library.
 *
 * The library holds no tensors.  Every buffer is owned by the caller and is
 * a DEVICE pointer unless stated otherwise; every call is asynchronous on
 * the stream it is given (a cudaStream_t passed as `pkv_stream_t`; NULL is
 * the legacy default stream).  A return value of PKV_OK means the work was
 * validated and launched; a fault inside a kernel surfaces at the caller's
 * next synchronisation, and index checks done on the device are reported
 * through pkv_get_device_error().  No call allocates device memory except
 * where stated.
 *
 * Data layout (nano-vLLM page "Maitriser les mecanismes cles de l'inference
 * des grands modeles avec nano-vLLM", section "Implementation du cache":
 * one layer's pool is torch.empty(2, num_blocks, block_size, kv_heads,
 * d_head)):
 *   k_cache, v_cache : [num_blocks][block_size][kv_heads][d_head] bf16,
 *                      contiguous, 16-byte aligned.  One slot (a token row)
 *                      is kv_heads * d_head contiguous elements.
 *   block_tables     : [num_seqs][max_blocks_per_seq] int32, row-major;
 *                      entry j of row s is the physical block holding logical
 *                      positions [16 j, 16 j + 16) of sequence s ("Cache KV,
 *                      attention et optimisation de l'inference", section
 *                      "PagedAttention KV cache comme memoire virtuelle").
 *   context_lens     : [num_seqs] int32, the number of tokens of each
 *                      sequence INCLUDING the ones appended in this step (the
 *                      cache is updated first and the new token attends to
 *                      itself: "Optimisation de l'inference", "Etape 1/2").
 *
 * Supported shapes: block_size 16; d_head 64 or 128; q_heads a multiple of
 * kv_heads with a group q_heads / kv_heads of 1, 2, 4, 8 or 16.  Anything
 * else returns PKV_EUNSUPPORTED without launching.
 */
#ifndef PAGEDKV_H_
#define PAGEDKV_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKV_OK = 0,
  PKV_EINVAL = -1,        /* null pointer, negative size, misaligned buffer or stride */
  PKV_EUNSUPPORTED = -2,  /* shape outside the supported set listed above */
  PKV_ECUDA = -3,         /* a CUDA runtime call or a kernel launch failed */
  PKV_ENOMEM = -4,        /* the workspace passed is smaller than required; host memory
                             ran out (block manager) */
  PKV_EDEVICE_CHECK = -5, /* pkv_get_last_device_error: a device-side check raised a bit */
  PKV_ETIMEOUT = -6,      /* pkv_get_last_device_error: a bounded device wait ran out */
  PKV_ESCRATCH_TOO_SMALL = -7, /* the no-allocation decode's fixed scratch cannot hold the plan */
  PKV_ENOBLOCKS = -8      /* block manager: fewer free blocks than needed; nothing changed */
} pkv_status;

/* Shape of one layer's K (and V) pool: [num_blocks][block_size][kv_heads][d_head]. */
typedef struct {
  int32_t num_blocks;
  int32_t block_size;
  int32_t kv_heads;
  int32_t d_head;
} pkv_cache_desc;

/* A cudaStream_t. */
typedef void* pkv_stream_t;

/* Bits of the device error word returned by pkv_get_device_error(). */
#define PKV_DEVERR_BAD_SLOT 0x1u        /* slot outside [-1, num_blocks*16): token skipped */
#define PKV_DEVERR_BAD_BLOCK_ID 0x2u    /* block id outside the pool: its rows read as 0 */
#define PKV_DEVERR_BAD_CONTEXT 0x4u     /* context_len < 0 or > 16*max_blocks_per_seq: clamped */
#define PKV_DEVERR_WAIT_TIMEOUT 0x8u    /* a bounded wait on an mbarrier ran out */
#define PKV_DEVERR_BAD_QUERY_RANGE 0x10u /* q_start not monotone or chunk longer than context */
#define PKV_DEVERR_TMEM_ALLOC 0x20u     /* tensor memory could not be allocated */
#define PKV_DEVERR_FP16_RANGE 0x40u     /* FP8 decode: a query value is outside f16's range */
#define PKV_DEVERR_DUPLICATE_SLOT 0x80u /* checked append: a slot named twice; nothing written */
#define PKV_DEVERR_PREFIX_MISMATCH 0x100u /* shared-prefix decode: a member's prefix is not its
                                             group's (or is out of range); decoded without it */

/*
 * pkv_kv_append -- scatter new K/V rows into the paged pools.
 *
 * Passage: nano-vLLM page, section "Ecriture dans le cache" (the store
 * kernel): for each new token t, slot = slot_mapping[t]; slot == -1 skips the
 * token; otherwise the token's kv_heads*d_head K elements are copied to row
 * `slot` of k_cache (block slot / 16, offset slot % 16) and likewise for V.
 * The copy is a bit copy.
 *
 *   k, v          : [num_tokens][kv_heads][d_head] bf16 rows; row t starts at
 *                   element t * k_tok_stride (resp. v_tok_stride), so views of
 *                   a fused QKV projection are accepted.  Base pointers and
 *                   strides must be 16-byte aligned (strides are in elements).
 *   slot_mapping  : [num_tokens] int64.  Two tokens with the same slot race
 *                   (the result is one of them; pkv_kv_append_checked
 *                   rejects such a mapping instead).
 *   k_cache, v_cache : pools described by `cache`, written in place.
 * Slots outside [-1, num_blocks*16) are skipped and set
 * PKV_DEVERR_BAD_SLOT.  num_tokens == 0 launches nothing.
 */
PKV_API int pkv_kv_append(const void* k, int64_t k_tok_stride, const void* v, int64_t v_tok_stride,
                  const int64_t* slot_mapping, int64_t num_tokens, void* k_cache,
                  void* v_cache, pkv_cache_desc cache, pkv_stream_t stream);

/*
 * pkv_kv_append_checked -- pkv_kv_append that rejects a slot mapping in
 * which two tokens name the same slot.  The pages' slot mapping gives each
 * new token its own cache row (nano-vLLM page, section "Ecriture dans le
 * cache"); two writers of one row would leave it undefined.  A device pass
 * marks every slot in [0, num_blocks*16) in a bitmap.  If any slot is
 * marked twice, PKV_DEVERR_DUPLICATE_SLOT is set and the append writes
 * nothing: the caches are left as they were.  Slots -1 (skip) and slots
 * outside the pool (skipped, PKV_DEVERR_BAD_SLOT) do not count as repeats.
 * No host synchronisation: the rejection happens on the stream.
 *   workspace : >= pkv_kv_append_checked_workspace_bytes(cache) device
 *               bytes, 256-byte aligned (PKV_ENOMEM if NULL or smaller);
 *               overwritten by every call, so calls that share it must be
 *               ordered on the GPU.
 * Other arguments and errors are those of pkv_kv_append.
 */
PKV_API size_t pkv_kv_append_checked_workspace_bytes(pkv_cache_desc cache);
PKV_API int pkv_kv_append_checked(const void* k, int64_t k_tok_stride, const void* v,
                                  int64_t v_tok_stride, const int64_t* slot_mapping,
                                  int64_t num_tokens, void* k_cache, void* v_cache,
                                  pkv_cache_desc cache, void* workspace, size_t ws_bytes,
                                  pkv_stream_t stream);

/*
 * How the split-K decode divides each sequence's pages (partition_blocks):
 *   > 0 (1..1024)        uniform partitions of that many 16-token blocks;
 *   PKV_SPLIT_UNIFORM    uniform partitions sized by the library from the
 *                        longest context and the device's SM count;
 *   PKV_SPLIT_BALANCED   a length-balanced work list (bf16 decode, at most
 *                        512 sequences): the kernel reads the actual
 *                        context lengths and cuts every (sequence, KV head)
 *                        pair's pages into runs of near-equal size, about
 *                        one wave of CTAs in all ("第 10 讲：推理（Inference）",
 *                        "核心概念与定义": FlashDecoding's split of long
 *                        contexts, here balanced on the real lengths);
 *   PKV_SPLIT_FLAT       the flat split (bf16 decode, at most 1024
 *                        sequences): a persistent grid of one CTA per SM
 *                        whose warps each stream one contiguous range of
 *                        the pages of all (sequence, KV head) pairs laid end
 *                        to end; the ranges differ by at most one page, and
 *                        a warp's page copies run on across the pairs of its
 *                        range, so the copy pipeline fills once per warp;
 *   0                    the library's choice: the flat split for 193 to
 *                        1024 (sequence, KV head) pairs at d_head 128 (and
 *                        for more pairs in 3 or more uniform partitions),
 *                        where it measured faster on GB300, else the uniform
 *                        partitions (the balanced list did not beat them at
 *                        any batch size: a small batch's time is the
 *                        decode's fixed cost more than the balance of its
 *                        waves).
 * The FP8 decode takes the flat split like the bf16 decode (PKV_SPLIT_FLAT,
 * or the library's choice, from 128 pairs over FP8 pages; the workspace of
 * the library's choice over bf16 pages covers it) and treats the other values
 * <= 0 as PKV_SPLIT_UNIFORM; the verification decode treats every value
 * <= 0 as PKV_SPLIT_UNIFORM; the shared-prefix decode takes the library's
 * choice for the sequences' own pages.
 */
#define PKV_SPLIT_BALANCED (-1)
#define PKV_SPLIT_UNIFORM (-2)
#define PKV_SPLIT_FLAT (-3)

/*
 * Decode plan: the partition size (in 16-token blocks) and the number of
 * partitions of the uniform split for these sizes, and the workspace the
 * bf16 decode needs with this partition_blocks (for the balanced list too,
 * when it is taken; this also covers the FP8 decode's uniform split).  The
 * plan depends on the current device.  Returns PKV_OK or PKV_EINVAL /
 * PKV_EUNSUPPORTED.
 */
PKV_API int pkv_decode_plan(int num_seqs, int q_heads, int kv_heads, int d_head, int max_context_len,
                    int partition_blocks, int* out_partition_blocks, int* out_num_parts,
                    size_t* out_workspace_bytes);

/* 1 when the bf16 decode with this partition_blocks takes the length-balanced
 * list, 0 when it takes the uniform split, or a negative pkv_status. */
PKV_API int pkv_decode_plan_uses_list(int num_seqs, int q_heads, int kv_heads, int d_head,
                                      int max_context_len, int partition_blocks);

/* 1 when the bf16 decode with this partition_blocks takes the flat split, 0
 * when it does not, or a negative pkv_status. */
PKV_API int pkv_decode_plan_uses_flat(int num_seqs, int q_heads, int kv_heads, int d_head,
                                      int max_context_len, int partition_blocks);

/* Workspace bytes pkv_paged_decode_attention needs with the library's choice
 * (0 when neither a list nor more than one partition is needed). */
PKV_API size_t pkv_decode_workspace_bytes(int num_seqs, int q_heads, int kv_heads, int d_head,
                                  int max_context_len);

/*
 * pkv_paged_decode_attention -- one query token per sequence attends over
 * its paged history (memory-bound decode step).
 *
 * Passages: "Optimisation de l'inference", section "Etape 2: Attention avec
 * KV Cache" (softmax(q K^T * scale) V, single query, no mask); "Cache KV,
 * attention et optimisation de l'inference", section "Etape 2: softmax en
 * carreaux" (online softmax: running max and sum, rescaled accumulator);
 * "第 10 讲：推理（Inference）", "核心概念与定义" (GQA: a group of query heads
 * shares one KV head; FlashDecoding named as the long-context method).
 *
 *   q            : [num_seqs][q_heads][d_head] bf16, contiguous.
 *   block_tables : [num_seqs][max_blocks_per_seq] int32.
 *   context_lens : [num_seqs] int32 (include this step's appended token).
 *   max_context_len : host-side bound on context_lens (>= every entry),
 *                  used to plan the split and size the workspace.  Tokens of
 *                  a longer sequence beyond the planned partitions are not
 *                  attended and PKV_DEVERR_BAD_CONTEXT is set.
 *   scale        : softmax scale, e.g. 1/sqrt(d_head).
 *   out          : [num_seqs][q_heads][d_head] float32 (not normalised to bf16).
 *   workspace    : device scratch of at least pkv_decode_workspace_bytes(...)
 *                  bytes, or NULL when that is 0; contents need no
 *                  initialisation and are overwritten.  Calls that share a
 *                  workspace must be ordered on the GPU.
 * Query head h uses KV head h / (q_heads / kv_heads).  A sequence with
 * context_len 0 yields zeros.  Block ids outside the pool read as zero rows
 * and set PKV_DEVERR_BAD_BLOCK_ID; context_len beyond 16*max_blocks_per_seq
 * is clamped and sets PKV_DEVERR_BAD_CONTEXT.  Returns PKV_ENOMEM if
 * ws_bytes is too small.
 */
PKV_API int pkv_paged_decode_attention(const void* q, int num_seqs, int q_heads, const void* k_cache,
                               const void* v_cache, pkv_cache_desc cache,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* context_lens, int max_context_len, float scale,
                               float* out, void* workspace, size_t ws_bytes,
                               pkv_stream_t stream);

/* Same as pkv_paged_decode_attention with an explicit split choice
 * (partition_blocks: a size in blocks, PKV_SPLIT_UNIFORM, PKV_SPLIT_BALANCED,
 * PKV_SPLIT_FLAT or 0 = library choice; see above). */
PKV_API int pkv_paged_decode_attention_ex(const void* q, int num_seqs, int q_heads, const void* k_cache,
                                  const void* v_cache, pkv_cache_desc cache,
                                  const int32_t* block_tables, int max_blocks_per_seq,
                                  const int32_t* context_lens, int max_context_len, float scale,
                                  float* out, void* workspace, size_t ws_bytes,
                                  int partition_blocks, pkv_stream_t stream);

/*
 * pkv_paged_decode_step -- one decode step: pkv_kv_append of each
 * sequence's new token, then pkv_paged_decode_attention, with the same
 * results (cache rows bit for bit, outputs bit for bit) and the append's time
 * hidden: the decode's CTAs start beside the append and only the loads of a
 * sequence's last page -- the one holding the appended token -- wait for it.
 * One new token per sequence: row s of k_new / v_new and slot_mapping[s]
 * belong to sequence s, and slot_mapping[s] must be -1 or the slot of its
 * position context_lens[s] - 1 (the usual decode step: the cache is updated,
 * then attended, "Optimisation de l'inference", "Etape 1/2").  A slot
 * elsewhere is still written but may be missed by the attention; it sets
 * PKV_DEVERR_BAD_SLOT.  Arguments as in pkv_kv_append and
 * pkv_paged_decode_attention (library's split choice; the workspace of
 * pkv_decode_workspace_bytes).
 */
PKV_API int pkv_paged_decode_step(const void* q, int num_seqs, int q_heads, const void* k_new,
                                  int64_t k_tok_stride, const void* v_new, int64_t v_tok_stride,
                                  const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                  pkv_cache_desc cache, const int32_t* block_tables,
                                  int max_blocks_per_seq, const int32_t* context_lens,
                                  int max_context_len, float scale, float* out, void* workspace,
                                  size_t ws_bytes, pkv_stream_t stream);

/*
 * pkv_paged_decode_attention_limited -- the decode on at most max_ctas CTAs,
 * leaving the other SMs to kernels on other streams (the continuous-batching
 * step runs a chunked prefill beside the decodes: nano-vLLM page, section
 * "Traitement par lots continu").  The length-balanced list of
 * PKV_SPLIT_BALANCED with about four runs per CTA; each CTA takes every
 * max_ctas-th run.  At most 512 sequences (PKV_EUNSUPPORTED beyond).
 * workspace: >= pkv_decode_limited_workspace_bytes(..., max_ctas) bytes,
 * 256-byte aligned (PKV_ENOMEM if smaller).  max_ctas >= 1 (PKV_EINVAL
 * otherwise).  Other arguments and errors are those of
 * pkv_paged_decode_attention.
 */
PKV_API size_t pkv_decode_limited_workspace_bytes(int num_seqs, int q_heads, int kv_heads,
                                                  int d_head, int max_context_len, int max_ctas);
PKV_API int pkv_paged_decode_attention_limited(const void* q, int num_seqs, int q_heads,
                                               const void* k_cache, const void* v_cache,
                                               pkv_cache_desc cache, const int32_t* block_tables,
                                               int max_blocks_per_seq,
                                               const int32_t* context_lens, int max_context_len,
                                               float scale, float* out, int max_ctas,
                                               void* workspace, size_t ws_bytes,
                                               pkv_stream_t stream);

/*
 * pkv_paged_decode_attention_bf16out -- pkv_paged_decode_attention_ex with a
 * bf16 output.  bf16 is inference's default type ("第 10 讲：推理（Inference）",
 * "核心概念与定义": bf16 as the inference default, 2 bytes per value in the
 * attention step's byte count), so the layer after attention reads bf16.
 * The arithmetic is the float32 path's; only the final store rounds each
 * value to the nearest bf16 (ties to even), so out equals the float32
 * output of pkv_paged_decode_attention_ex rounded to bf16, bit for bit.
 *   out : [num_seqs][q_heads][d_head] bf16, 2-byte aligned (8-byte
 *         alignment lets the split-K merge store four values at once).
 * Other arguments, the workspace and the errors are those of
 * pkv_paged_decode_attention_ex.
 */
PKV_API int pkv_paged_decode_attention_bf16out(const void* q, int num_seqs, int q_heads,
                                               const void* k_cache, const void* v_cache,
                                               pkv_cache_desc cache,
                                               const int32_t* block_tables,
                                               int max_blocks_per_seq,
                                               const int32_t* context_lens, int max_context_len,
                                               float scale, void* out, void* workspace,
                                               size_t ws_bytes, int partition_blocks,
                                               pkv_stream_t stream);

/*
 * pkv_paged_prefill_attention -- chunked prefill: each sequence's new query
 * tokens attend over its paged context (the continuous-batching step in which
 * new prompt chunks join running decodes).  Runs on the tcgen05 tensor cores.
 *
 * Passages: "Optimisation de l'inference", section "Etape 2: Attention avec
 * KV Cache" (softmax(q K^T * scale + mask) V; for more than one query the
 * mask is triu(ones(Tq, Tk), k = Tk - Tq + 1), i.e. bottom-right aligned);
 * "Cache KV, attention et optimisation de l'inference", section "Attention a
 * la lumiere" (FlashAttention tiling: a query tile stays on chip while K/V
 * tiles stream by with a running max and sum).
 *
 *   q            : [total_q][q_heads][d_head] bf16, contiguous; the rows
 *                  q_start[s] .. q_start[s+1]-1 are the chunk of sequence s.
 *   q_start      : [num_seqs + 1] int32, non-decreasing, q_start[num_seqs] <= total_q.
 *   max_q_len    : host bound on q_start[s+1] - q_start[s] (sizes the grid).
 *   context_lens : [num_seqs] int32, INCLUDING the chunk (its K/V must have
 *                  been appended first); the chunk is the last n tokens.
 *   causal       : nonzero = query i of a chunk of n sees keys
 *                  0 .. context_len - n + i; zero = every query sees the
 *                  whole context.
 *   out          : [total_q][q_heads][d_head] float32, 16-byte aligned; rows
 *                  outside every chunk are not written.
 * A chunk longer than its context, a chunk longer than max_q_len, a
 * non-monotone q_start or a context beyond the block table rejects that
 * sequence: none of its rows is written and PKV_DEVERR_BAD_QUERY_RANGE is set
 * (pkv_get_last_device_error returns PKV_EDEVICE_CHECK).  No workspace is
 * needed.
 */
PKV_API int pkv_paged_prefill_attention(const void* q, const int32_t* q_start, int num_seqs,
                                        int total_q, int max_q_len, int q_heads,
                                        const void* k_cache, const void* v_cache,
                                        pkv_cache_desc cache, const int32_t* block_tables,
                                        int max_blocks_per_seq, const int32_t* context_lens,
                                        int causal, float scale, float* out,
                                        pkv_stream_t stream);

/*
 * pkv_paged_prefill_attention_ex -- pkv_paged_prefill_attention with a
 * workspace that buys a faster kernel.  The V pages the chunks' sequences
 * use are first converted to f16 in the workspace (page j of sequence s to
 * scratch block s * max_blocks_per_seq + j); the tensor-core prefill then
 * reads K from the pool and V from the workspace and feeds P to the P V
 * product as one f16 operand (rounding error <= 2^-11 relative, so the
 * output moves by at most 2^-11 times the largest |V| a row attends to),
 * instead of the bf16 hi + lo pair the plain entry point needs -- one third
 * less tensor-core work for one bf16 read and one f16 write per V element of
 * those pages.  The conversion is exact for |v| in [2^-14, 65504]; smaller
 * values become f16 subnormals (absolute error < 2^-25); a value of
 * magnitude 65520 or more overflows and sets PKV_DEVERR_FP16_RANGE.  The
 * error bound scales with V: an output element is off by at most
 * 2^-10 * max|V| (measured 8.7e-5 * max|V|), so the absolute 2e-3 of the
 * tests holds while |V| stays below about 20; for larger V use
 * pkv_paged_prefill_attention (P as bf16 hi + lo, ~2^-17).  The
 * same pass ranks the sequences by context length, and the prefill runs
 * each sequence's tiles together, longest context first (a dispatch order
 * only: the result does not depend on it).
 * workspace: >= pkv_paged_prefill_workspace_bytes(num_seqs,
 * max_blocks_per_seq, kv_heads, d_head) device bytes, 256-byte aligned
 * (PKV_ENOMEM if smaller); NULL runs pkv_paged_prefill_attention.
 */
PKV_API size_t pkv_paged_prefill_workspace_bytes(int num_seqs, int max_blocks_per_seq,
                                                 int kv_heads, int d_head);
PKV_API int pkv_paged_prefill_attention_ex(const void* q, const int32_t* q_start, int num_seqs,
                                           int total_q, int max_q_len, int q_heads,
                                           const void* k_cache, const void* v_cache,
                                           pkv_cache_desc cache, const int32_t* block_tables,
                                           int max_blocks_per_seq, const int32_t* context_lens,
                                           int causal, float scale, float* out, void* workspace,
                                           size_t ws_bytes, pkv_stream_t stream);

/*
 * pkv_paged_prefill_attention_limited -- pkv_paged_prefill_attention_ex on at
 * most max_ctas SMs, leaving the others to kernels on other streams.  The
 * continuous-batching step (nano-vLLM page, section "Traitement par lots
 * continu"; "第 10 讲：推理（Inference）", "关键要点": iteration-level
 * scheduling and selective batching) runs chunked prefills next to running
 * decodes.  The prefill is bound by the tensor cores and the decode by HBM,
 * so a decode launched on another stream after this call runs on the
 * remaining SMs at the same time instead of after it.
 * Same result as pkv_paged_prefill_attention_ex (bit for bit: the same
 * tiles in the same arithmetic); max_ctas persistent CTAs take the
 * (sequence x KV head, query tile) items from a counter in the workspace,
 * in the dispatch order of pkv_paged_prefill_attention_ex.  max_ctas >= 1 (PKV_EINVAL otherwise); a workspace of
 * pkv_paged_prefill_workspace_bytes(...) bytes is required (PKV_ENOMEM if
 * NULL or smaller).  Calls that share a workspace must not overlap.
 */
PKV_API int pkv_paged_prefill_attention_limited(const void* q, const int32_t* q_start,
                                                int num_seqs, int total_q, int max_q_len,
                                                int q_heads, const void* k_cache,
                                                const void* v_cache, pkv_cache_desc cache,
                                                const int32_t* block_tables,
                                                int max_blocks_per_seq,
                                                const int32_t* context_lens, int causal,
                                                float scale, float* out, int max_ctas,
                                                void* workspace, size_t ws_bytes,
                                                pkv_stream_t stream);

/*
 * pkv_mixed_step_attention -- the attention of one continuous-batching step
 * in a single persistent launch: the chunked prefill of num_prefill new
 * prompt chunks and the decode of num_decode running sequences, over the
 * same K/V pools ("第 10 讲：推理（Inference）", "核心概念与定义": continuous
 * batching and selective batching -- attention per sequence, every request of
 * the step in one batch; nano-vLLM page, section "Priorité au
 * pré-remplissage").  Every SM takes items from one work list: query tiles of
 * the chunks (tensor cores) and length-balanced runs of the decodes (HBM),
 * interleaved so that SMs free of one kind of work take the other; the
 * library sizes the split from the actual lengths, not from a caller's
 * choice.  Results: out_prefill as pkv_paged_prefill_attention_ex (bit for
 * bit: the same tile arithmetic, P as one f16 operand -- see there for the
 * accuracy and V's range), out_decode as pkv_paged_decode_attention with
 * PKV_SPLIT_BALANCED (within the decode's tolerance: the runs differ).
 * Before the call, the K/V of every new token (chunks and decode tokens)
 * must be appended.
 *   prefill part : q_prefill [total_q][q_heads][d_head] bf16, q_start [num_prefill + 1],
 *                  prefill_block_tables [num_prefill][prefill_max_blocks],
 *                  prefill_context_lens [num_prefill], causal -- as in
 *                  pkv_paged_prefill_attention; out_prefill [total_q][q_heads][d_head] fp32.
 *   decode part  : q_decode [num_decode][q_heads][d_head] bf16 (num_decode <= 512),
 *                  decode_block_tables [num_decode][decode_max_blocks],
 *                  decode_context_lens [num_decode], max_decode_context_len
 *                  (host bound) -- as in pkv_paged_decode_attention;
 *                  out_decode [num_decode][q_heads][d_head] fp32, 16-byte aligned.
 *   workspace    : >= pkv_mixed_step_workspace_bytes(...) device bytes,
 *                  256-byte aligned (PKV_ENOMEM if smaller); overwritten by
 *                  every call, so calls that share it must not overlap.
 * Both parts must be non-empty (PKV_EINVAL otherwise; each separate entry
 * point serves one part alone).  Errors and device checks are those of the
 * two separate calls.
 */
PKV_API size_t pkv_mixed_step_workspace_bytes(int num_prefill, int prefill_max_blocks,
                                              int num_decode, int q_heads, int kv_heads,
                                              int d_head, int max_decode_context_len);
PKV_API int pkv_mixed_step_attention(const void* q_prefill, const int32_t* q_start,
                                     int num_prefill, int total_q, int max_q_len,
                                     const int32_t* prefill_block_tables, int prefill_max_blocks,
                                     const int32_t* prefill_context_lens, int causal,
                                     const void* q_decode, int num_decode,
                                     const int32_t* decode_block_tables, int decode_max_blocks,
                                     const int32_t* decode_context_lens,
                                     int max_decode_context_len, int q_heads,
                                     const void* k_cache, const void* v_cache,
                                     pkv_cache_desc cache, float scale, float* out_prefill,
                                     float* out_decode, void* workspace, size_t ws_bytes,
                                     pkv_stream_t stream);

/* pkv_mixed_step_attention with decode prefix groups and the work list's
 * interleave as parameters.
 *   decode_group_start, decode_group_prefix_blocks, num_groups,
 *   max_group_size, max_prefix_blocks: prefix groups of the decodes exactly
 *     as in pkv_paged_decode_attention_prefix_groups (device arrays; members
 *     checked against their leader; num_groups 0 = none).  The list then
 *     starts with each group's prefix items -- its members' queries against
 *     its prefix on the tensor cores -- and the decode runs cover only the
 *     members' own pages; the merge folds the prefix part in.
 *   prefill_span_permille: the prefill items are spread evenly over the first
 *     prefill_span_permille per mille of the rest of the list (1..1000), the
 *     remainder holding decode runs only; 0 = the library's value.  The
 *     results do not depend on it (the same items, another order).
 * workspace: >= pkv_mixed_step_groups_workspace_bytes(..., num_groups). */
PKV_API size_t pkv_mixed_step_groups_workspace_bytes(int num_prefill, int prefill_max_blocks,
                                                     int num_decode, int q_heads, int kv_heads,
                                                     int d_head, int max_decode_context_len,
                                                     int num_groups);
PKV_API int pkv_mixed_step_attention_ex(const void* q_prefill, const int32_t* q_start,
                                        int num_prefill, int total_q, int max_q_len,
                                        const int32_t* prefill_block_tables,
                                        int prefill_max_blocks,
                                        const int32_t* prefill_context_lens, int causal,
                                        const void* q_decode, int num_decode,
                                        const int32_t* decode_block_tables, int decode_max_blocks,
                                        const int32_t* decode_context_lens,
                                        int max_decode_context_len, int q_heads,
                                        const void* k_cache, const void* v_cache,
                                        pkv_cache_desc cache, float scale, float* out_prefill,
                                        float* out_decode, const int32_t* decode_group_start,
                                        const int32_t* decode_group_prefix_blocks,
                                        int num_groups, int max_group_size,
                                        int max_prefix_blocks, void* workspace, size_t ws_bytes,
                                        int prefill_span_permille, pkv_stream_t stream);

/*
 * pkv_paged_prefill_attention_bf16out -- the chunked prefill with a bf16
 * output (bf16 as the inference default: "第 10 讲：推理（Inference）",
 * "核心概念与定义").  With a workspace it is pkv_paged_prefill_attention_ex,
 * with workspace NULL pkv_paged_prefill_attention; the epilogue rounds each
 * value of O / l (ties to even) instead of storing float32, so out equals
 * that entry point's float32 output rounded to bf16, bit for bit.
 *   out : [total_q][q_heads][d_head] bf16, 16-byte aligned; rows outside
 *         every chunk are not written.
 * Other arguments, the workspace and the errors are those of
 * pkv_paged_prefill_attention_ex.
 */
PKV_API int pkv_paged_prefill_attention_bf16out(const void* q, const int32_t* q_start,
                                                int num_seqs, int total_q, int max_q_len,
                                                int q_heads, const void* k_cache,
                                                const void* v_cache, pkv_cache_desc cache,
                                                const int32_t* block_tables,
                                                int max_blocks_per_seq,
                                                const int32_t* context_lens, int causal,
                                                float scale, void* out, void* workspace,
                                                size_t ws_bytes, pkv_stream_t stream);

/*
 * pkv_paged_decode_attention_prefix_groups -- the same result as
 * pkv_paged_decode_attention when groups of sequences share their first
 * pages: the same physical blocks for a system prompt stored once, or for
 * the forks of one prompt ("Optimisation de l'inference", section
 * "PageAtention": many requests on one system prompt's pages; nano-vLLM
 * page, section "Implementation du cache": prefix blocks shared through the
 * chained hash).  Each group's prefix is read once for all its members
 * instead of once per member:
 *   0. a device pass checks every member: its first prefix blocks must be
 *      the group leader's ids (the leader is the group's first sequence) and
 *      its context must hold the prefix; a member that fails -- or whose
 *      group's prefix length is out of range -- is decoded over its whole
 *      context instead, and PKV_DEVERR_PREFIX_MISMATCH is set;
 *   1. each group's member queries attend the group's prefix keys
 *      (non-causal) on the tensor cores, giving a normalised output and
 *      log-sum-exp per (sequence, head);
 *   2. each sequence's own pages after its prefix go through the split-K
 *      decode;
 *   3. the log-sum-exp merge combines both parts.
 *   group_start        : [num_groups + 1] int32 device, non-decreasing: group g is
 *                        sequences group_start[g] .. group_start[g+1] - 1 (the batch
 *                        is ordered by group); sequences outside every group
 *                        have no shared prefix.
 *   group_prefix_blocks: [num_groups] int32 device: group g's prefix in 16-token
 *                        blocks, 1 .. max_prefix_blocks.
 *   max_group_size     : host bound on group_start[g+1] - group_start[g].
 *   max_prefix_blocks  : host bound on group_prefix_blocks.
 * workspace: >= pkv_decode_prefix_groups_workspace_bytes(...) bytes, 256-byte
 * aligned.  Other arguments and errors are those of
 * pkv_paged_decode_attention.
 *
 * pkv_paged_decode_attention_shared_prefix -- the case of one group of
 * every sequence, whose prefix is the first prefix_blocks ids of row 0;
 * workspace: pkv_decode_shared_prefix_workspace_bytes(...) bytes.
 */
PKV_API size_t pkv_decode_prefix_groups_workspace_bytes(int num_seqs, int q_heads, int kv_heads,
                                                       int d_head, int max_context_len,
                                                       int num_groups);
PKV_API int pkv_paged_decode_attention_prefix_groups(
    const void* q, int num_seqs, int q_heads, const void* k_cache, const void* v_cache,
    pkv_cache_desc cache, const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* context_lens, int max_context_len, const int32_t* group_start,
    const int32_t* group_prefix_blocks, int num_groups, int max_group_size,
    int max_prefix_blocks, float scale, float* out, void* workspace, size_t ws_bytes,
    pkv_stream_t stream);

PKV_API size_t pkv_decode_shared_prefix_workspace_bytes(int num_seqs, int q_heads, int kv_heads,
                                                        int d_head, int max_context_len,
                                                        int prefix_blocks);

PKV_API int pkv_paged_decode_attention_shared_prefix(
    const void* q, int num_seqs, int q_heads, const void* k_cache, const void* v_cache,
    pkv_cache_desc cache, const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* context_lens, int max_context_len, int prefix_blocks, float scale, float* out,
    void* workspace, size_t ws_bytes, pkv_stream_t stream);

/*
 * pkv_paged_verify_attention -- multi-query decode, the verification step of
 * speculative decoding ("Cache KV, attention et optimisation de
 * l'inference", section "Decodage speculatif": guess several next tokens
 * cheaply, then check them all in one pass).  Each sequence has q_len query
 * tokens, already appended, as the last q_len positions of its context:
 * token t (0 <= t < q_len) sits at position context_len - q_len + t and
 * attends over keys 0 .. context_len - q_len + t (the bottom-right causal
 * mask of a q_len-token prefill chunk).
 *   q   : [num_seqs][q_len][q_heads][d_head] bf16, contiguous.
 *   out : [num_seqs][q_len][q_heads][d_head] fp32.
 * (q_heads / kv_heads) * q_len must be <= 32 (e.g. 4 drafted tokens with a
 * GQA group of 8), else PKV_EUNSUPPORTED.  The K/V bytes of a (sequence, KV
 * head) are read once for all its query tokens and heads; long contexts are
 * split as in the decode (same plan for the given partition_blocks, 0 =
 * library choice), with a workspace of
 * pkv_verify_workspace_bytes(...) device bytes (0: none needed).  A context
 * shorter than q_len sets PKV_DEVERR_BAD_QUERY_RANGE; tokens placed before
 * position 0 see no key and return zeros.
 */
PKV_API size_t pkv_verify_workspace_bytes(int num_seqs, int q_len, int q_heads, int kv_heads,
                                          int d_head, int max_context_len, int partition_blocks);
PKV_API int pkv_paged_verify_attention(const void* q, int num_seqs, int q_len, int q_heads,
                                       const void* k_cache, const void* v_cache,
                                       pkv_cache_desc cache, const int32_t* block_tables,
                                       int max_blocks_per_seq, const int32_t* context_lens,
                                       int max_context_len, float scale, float* out,
                                       void* workspace, size_t ws_bytes, int partition_blocks,
                                       pkv_stream_t stream);

/* pkv_paged_verify_attention with a bf16 output: the float32 result rounded
 * to the nearest bf16 (ties to even) in the final store, bit for bit (see
 * pkv_paged_decode_attention_bf16out).  out: [num_seqs][q_len][q_heads]
 * [d_head] bf16, 2-byte aligned. */
PKV_API int pkv_paged_verify_attention_bf16out(const void* q, int num_seqs, int q_len,
                                               int q_heads, const void* k_cache,
                                               const void* v_cache, pkv_cache_desc cache,
                                               const int32_t* block_tables,
                                               int max_blocks_per_seq,
                                               const int32_t* context_lens, int max_context_len,
                                               float scale, void* out, void* workspace,
                                               size_t ws_bytes, int partition_blocks,
                                               pkv_stream_t stream);

/*
 * FP8 KV cache.  The pages name FP8 KV caches as the way to halve decode's
 * KV bytes ("Cache KV, attention et optimisation de l'inference", section
 * "Utilisez-le": --kv-cache-dtype fp8; "第 10 讲：推理（Inference）": fewer
 * bits, fewer bytes) without fixing a format.  Here: pools of e4m3 codes
 * (one byte each, same [num_blocks][16][kv_heads][d_head] layout) with one
 * float32 scale per pool; a code c stands for e4m3(c) * scale.
 *
 * pkv_kv_append_fp8 -- as pkv_kv_append, but each element is stored as
 * e4m3(float32(x) * (1 / scale)), rounded to nearest even, finite overflow
 * saturating to +-448.  k/v are bf16 rows; scales must be positive and
 * finite; kv_heads * d_head must be a multiple of 16.
 */
PKV_API int pkv_kv_append_fp8(const void* k, int64_t k_tok_stride, const void* v,
                              int64_t v_tok_stride, const int64_t* slot_mapping,
                              int64_t num_tokens, void* k_cache, void* v_cache,
                              pkv_cache_desc cache, float k_scale, float v_scale,
                              pkv_stream_t stream);

/*
 * pkv_paged_decode_attention_fp8 -- pkv_paged_decode_attention over FP8
 * pools: the result is the attention of the dequantized cache
 * (K = k_scale * e4m3(k_cache), V = v_scale * e4m3(v_cache)).  d_head must
 * be 128.  Same plan and workspace as the bf16 decode (pkv_decode_plan);
 * partition_blocks 0 = library choice, PKV_SPLIT_FLAT = the flat split, other
 * values <= 0 = uniform partitions.  Query values must fit f16's range
 * (|q| < 65520), else PKV_DEVERR_FP16_RANGE is set.  P enters the P V
 * product as one f16 operand: an output element is off by at most
 * 2^-10 * max|V| of the dequantized V (measured 5.3e-5 * max|V|).
 */
PKV_API int pkv_paged_decode_attention_fp8(const void* q, int num_seqs, int q_heads,
                                           const void* k_cache, const void* v_cache,
                                           pkv_cache_desc cache, const int32_t* block_tables,
                                           int max_blocks_per_seq, const int32_t* context_lens,
                                           int max_context_len, float scale, float k_scale,
                                           float v_scale, float* out, void* workspace,
                                           size_t ws_bytes, int partition_blocks,
                                           pkv_stream_t stream);

/* pkv_paged_decode_attention_fp8 with a bf16 output: the float32 result
 * rounded to the nearest bf16 (ties to even) in the final store, bit for bit
 * (see pkv_paged_decode_attention_bf16out).  out: [num_seqs][q_heads][128]
 * bf16, 2-byte aligned. */
PKV_API int pkv_paged_decode_attention_fp8_bf16out(const void* q, int num_seqs, int q_heads,
                                                   const void* k_cache, const void* v_cache,
                                                   pkv_cache_desc cache,
                                                   const int32_t* block_tables,
                                                   int max_blocks_per_seq,
                                                   const int32_t* context_lens,
                                                   int max_context_len, float scale,
                                                   float k_scale, float v_scale, void* out,
                                                   void* workspace, size_t ws_bytes,
                                                   int partition_blocks, pkv_stream_t stream);

/*
 * pkv_paged_prefill_attention_fp8 -- pkv_paged_prefill_attention over FP8
 * pools: the attention of the dequantized cache, as above.  The pages a
 * chunk's sequence uses (its first ceil(context_len / 16) block-table
 * entries) are first widened in the workspace, K to bf16 and V to f16 --
 * exact, every e4m3 value is a bf16 and an f16 value -- and the tensor-core
 * prefill then runs on them with k_scale folded into the softmax scale,
 * v_scale into the output, and P as one f16 operand (see
 * pkv_paged_prefill_attention_ex).  That
 * costs one FP8 read and one bf16 write per cached element of those pages on
 * top of the bf16 prefill.  d_head 64 or 128.
 * workspace: >= pkv_paged_prefill_attention_fp8_workspace_bytes(num_seqs,
 * max_blocks_per_seq, kv_heads, d_head) device bytes (PKV_ENOMEM otherwise);
 * its contents on entry do not matter.  Out-of-range block ids read as zeros
 * and set PKV_DEVERR_BAD_BLOCK_ID.
 */
PKV_API size_t pkv_paged_prefill_attention_fp8_workspace_bytes(int num_seqs,
                                                               int max_blocks_per_seq,
                                                               int kv_heads, int d_head);
PKV_API int pkv_paged_prefill_attention_fp8(const void* q, const int32_t* q_start, int num_seqs,
                                            int total_q, int max_q_len, int q_heads,
                                            const void* k_cache, const void* v_cache,
                                            pkv_cache_desc cache, const int32_t* block_tables,
                                            int max_blocks_per_seq, const int32_t* context_lens,
                                            int causal, float scale, float k_scale, float v_scale,
                                            float* out, void* workspace, size_t ws_bytes,
                                            pkv_stream_t stream);

/*
 * pkv_paged_prefill_attention_fp8_limited -- pkv_paged_prefill_attention_fp8
 * on at most max_ctas SMs (persistent CTAs taking query tiles from a counter
 * in the workspace), leaving the other SMs to a decode launched on another
 * stream, as pkv_paged_prefill_attention_limited does for bf16 pools.  Same
 * result bit for bit.  max_ctas >= 1 (PKV_EINVAL otherwise); the workspace
 * as for pkv_paged_prefill_attention_fp8.  Calls that share a workspace must
 * not overlap.
 */
PKV_API int pkv_paged_prefill_attention_fp8_limited(const void* q, const int32_t* q_start,
                                                    int num_seqs, int total_q, int max_q_len,
                                                    int q_heads, const void* k_cache,
                                                    const void* v_cache, pkv_cache_desc cache,
                                                    const int32_t* block_tables,
                                                    int max_blocks_per_seq,
                                                    const int32_t* context_lens, int causal,
                                                    float scale, float k_scale, float v_scale,
                                                    float* out, int max_ctas, void* workspace,
                                                    size_t ws_bytes, pkv_stream_t stream);

/*
 * Decode for callers that cannot allocate device memory.  The pages have no
 * counterpart to this entry point; it exists for callers that are handed
 * device buffers but may not call cudaMalloc (a fixed, pre-reserved memory
 * budget with no allocator, a plug-in inside another runtime, a serving loop
 * that must never allocate mid-step).
 *
 * Same computation and arguments as pkv_paged_decode_attention_ex, but the
 * split-K scratch is a 32 MiB array compiled into the library
 * (pkv_noalloc_scratch_bytes()), held by every GPU that loads the library
 * until the process exits.  No call allocates or frees memory.  The first
 * call on a device looks up the array's device address (make it before any
 * stream capture).  All calls share the array: calls whose work overlaps on
 * the GPU race on it, so order them on one stream.  Nothing in it needs to
 * start at zero.  Returns PKV_ESCRATCH_TOO_SMALL when the plan for these
 * sizes (pkv_decode_plan's workspace bytes) exceeds the array; a larger
 * partition_blocks needs less scratch.
 */
PKV_API size_t pkv_noalloc_scratch_bytes(void);

PKV_API int pkv_paged_decode_attention_noalloc(const void* q, int num_seqs, int q_heads,
                                               const void* k_cache, const void* v_cache,
                                               pkv_cache_desc cache,
                                               const int32_t* block_tables,
                                               int max_blocks_per_seq,
                                               const int32_t* context_lens, int max_context_len,
                                               float scale, float* out, int partition_blocks,
                                               pkv_stream_t stream);

/*
 * pkv_get_last_device_error -- the checked-mode status of the work queued on
 * `stream` so far.  The kernels never trap: a bad index is skipped and a
 * stuck wait gives up, each raising a PKV_DEVERR_* bit in the current
 * device's error words.  This call queues a one-thread kernel on `stream`
 * that takes those words and resets them to 0 in one atomic exchange per
 * word, copies the OR back and synchronises `stream` only (not the device).
 * Returns PKV_OK when no bit was raised, PKV_ETIMEOUT when a bounded wait ran
 * out (PKV_DEVERR_WAIT_TIMEOUT), PKV_EDEVICE_CHECK for any other bit, and
 * PKV_ECUDA when the launch, the copy or the synchronisation failed (e.g. a
 * stream being captured into a graph).  The words belong to the device, not
 * to the stream: bits raised by kernels of other streams that finished
 * before the exchange are reported (and cleared) too; a bit raised after it
 * stays for the next query.  pkv_get_last_device_error_bits also stores the
 * bits in *word (NULL allowed).  Host threads' calls are serialised.
 */
PKV_API int pkv_get_last_device_error(pkv_stream_t stream);
PKV_API int pkv_get_last_device_error_bits(pkv_stream_t stream, unsigned int* word);

/*
 * Read the device error word of the current device (an OR of the
 * PKV_DEVERR_* bits raised by kernels since the last clear).  Synchronises
 * the device.  clear != 0 resets the word to 0.  Returns PKV_OK or PKV_ECUDA.
 */
PKV_API int pkv_get_device_error(unsigned int* word, int clear);

/*
 * Failure detection without a fault.  Every kernel waits on its mbarriers
 * (copies landed, MMAs done) through one bounded wait: after
 * pkv_wait_poll_limit() polls it gives up, sets PKV_DEVERR_WAIT_TIMEOUT,
 * waits (again bounded) for its own copies in flight and returns, so a
 * stuck copy or MMA ends in an error the host reads instead of a hang.
 * pkv_wait_timeout_probe runs that same wait in a one-thread kernel on a
 * barrier phase that never completes, with `polls` (1 ..
 * pkv_wait_poll_limit()) as the limit: the wait runs out, the timeout bit
 * is set and the kernel returns.  cycles (device pointer, 8-byte aligned,
 * or NULL) receives the clock64 cycles the wait took.  PKV_EINVAL for polls
 * out of range.
 */
PKV_API uint32_t pkv_wait_poll_limit(void);
PKV_API int pkv_wait_timeout_probe(uint32_t polls, unsigned long long* cycles,
                                   pkv_stream_t stream);

/* Human-readable name of a pkv_status value (static string). */
PKV_API const char* pkv_status_string(int status);

/* Library version as 10000*major + 100*minor + patch. */
PKV_API int pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H_ */
