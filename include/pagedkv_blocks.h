/*
 * pagedkv_blocks.h -- host block manager of a paged KV cache, and the device
 * copy that backs its copy-on-write.
 *
 * The block manager is plain host code: it owns no device memory and never
 * touches tensor data.  It hands out physical block ids of a pool the caller
 * allocated once at start (nano-vLLM page "Maitriser les mecanismes cles de
 * l'inference des grands modeles avec nano-vLLM", section "Implementation du
 * cache"), keeps each sequence's block table, and produces the slot mapping
 * and block tables that pkv_kv_append, pkv_paged_decode_attention and
 * pkv_paged_prefill_attention take (pagedkv.h).
 *
 * Policy (the pages describe the mechanism; the policy choices are this
 * library's, stated here so that callers can rely on them):
 *   - Free list: first in, first out, initially 0 .. num_blocks-1; a freed
 *     sequence returns its blocks last-to-first ("Cache KV, attention et
 *     optimisation de l'inference": fixed 16-token pages anywhere in memory,
 *     a free list that finished sequences return their blocks to).
 *   - Prefix sharing: every full block carries a chained hash, FNV-1a 64-bit
 *     continued from the previous block's hash over the block's int32 token
 *     ids (little-endian bytes), starting from the FNV offset basis; a block
 *     whose hash and token ids match is shared, and a reference count keeps
 *     it alive (nano-vLLM page, "Implementation du cache").  Only a leading
 *     run of full prompt blocks is shared, never the block that holds the
 *     last prompt token.  A freed block keeps its cached content, and can be
 *     hit again, until it is handed out for new content.
 *   - Copy-on-write: appending to a sequence whose last block is partly
 *     filled and shared (after pkv_bm_fork, or when a partial block is
 *     shared) first moves the sequence to a new block and reports the pair
 *     (old, new); the caller copies it with pkv_copy_blocks before the
 *     appended rows are written ("Cache KV, attention...", section
 *     "PageAtention": the shared system prompt is stored once).
 *   - An operation that needs more free blocks than the pool has changes
 *     nothing and returns PKV_ENOBLOCKS.
 *
 * A manager is not thread-safe: calls on one handle must be serialised by the
 * caller.  Host pointers below are HOST memory unless marked "device".
 */
#ifndef PAGEDKV_BLOCKS_H_
#define PAGEDKV_BLOCKS_H_

#include "pagedkv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_block_manager pkv_block_manager;

/* A pool of num_blocks blocks of block_size tokens, all free.  *out receives
 * the handle (NULL on error).  PKV_EINVAL for non-positive sizes or a NULL
 * out; PKV_ENOMEM if host memory runs out. */
PKV_API int pkv_bm_create(int32_t num_blocks, int32_t block_size, pkv_block_manager** out);

/* Frees the handle and every sequence in it (NULL is ignored). */
PKV_API void pkv_bm_destroy(pkv_block_manager* bm);

/* Registers sequence seq_id with its prompt token_ids[0 .. num_tokens) and
 * gives it blocks for all of them.  *num_cached_tokens (may be NULL) receives
 * how many leading prompt tokens already sit in shared blocks: the caller
 * computes and appends K/V only for positions [*num_cached_tokens,
 * num_tokens), whose slots pkv_bm_slots returns.  PKV_EINVAL if seq_id is
 * already registered or num_tokens < 0 (token_ids may be NULL when 0);
 * PKV_ENOBLOCKS if the pool is short. */
PKV_API int pkv_bm_add_sequence(pkv_block_manager* bm, int64_t seq_id, const int32_t* token_ids,
                                int32_t num_tokens, int32_t* num_cached_tokens);

/* Reserves positions [len, len + num_tokens) of seq_id for the tokens
 * token_ids and writes their slots (block * block_size + offset) to
 * slots[0 .. num_tokens).  Copy-on-write pairs (src, dst) go to
 * copy_pairs[2 i], copy_pairs[2 i + 1] for i < *num_copies (at most one pair
 * per call); max_copies is the room in copy_pairs, in pairs.  Blocks that
 * become full are hashed and become shareable.  PKV_EINVAL for an unknown
 * seq_id, a NULL pointer, num_tokens < 0, or max_copies too small for the
 * copy the call needs (nothing is changed then); PKV_ENOBLOCKS if the pool is
 * short. */
PKV_API int pkv_bm_append_tokens(pkv_block_manager* bm, int64_t seq_id, const int32_t* token_ids,
                                 int32_t num_tokens, int64_t* slots, int32_t* copy_pairs,
                                 int32_t max_copies, int32_t* num_copies);

/* child becomes a copy of parent that shares all of its blocks (each block's
 * reference count goes up by one); no block is copied until one of them
 * appends into a shared partial block.  PKV_EINVAL if parent is unknown or
 * child already exists. */
PKV_API int pkv_bm_fork(pkv_block_manager* bm, int64_t parent, int64_t child);

/* Drops seq_id; blocks whose count reaches zero go to the back of the free
 * list, last block first.  PKV_EINVAL for an unknown seq_id. */
PKV_API int pkv_bm_free_sequence(pkv_block_manager* bm, int64_t seq_id);

/* Slots of positions [start, start + count) of seq_id into slots[0 .. count).
 * PKV_EINVAL if the range is outside [0, len). */
PKV_API int pkv_bm_slots(const pkv_block_manager* bm, int64_t seq_id, int32_t start, int32_t count,
                         int64_t* slots);

/* Number of tokens of seq_id into *len. PKV_EINVAL for an unknown seq_id. */
PKV_API int pkv_bm_seq_len(const pkv_block_manager* bm, int64_t seq_id, int32_t* len);

/* The block table of seq_id: its block ids into blocks[0 .. *num_blocks) if
 * they fit in cap (PKV_EINVAL otherwise, with *num_blocks set to the count
 * needed). */
PKV_API int pkv_bm_block_table(const pkv_block_manager* bm, int64_t seq_id, int32_t* blocks,
                               int32_t cap, int32_t* num_blocks);

/* Batch export in the layout the attention calls take: row s of
 * block_tables[num_seqs][max_blocks_per_seq] (int32, row-major) receives the
 * blocks of seq_ids[s], padded with 0, and context_lens[s] its length.
 * PKV_EINVAL for an unknown id, or a sequence with more blocks than
 * max_blocks_per_seq (nothing is written then). */
PKV_API int pkv_bm_block_tables(const pkv_block_manager* bm, const int64_t* seq_ids,
                                int32_t num_seqs, int32_t* block_tables,
                                int32_t max_blocks_per_seq, int32_t* context_lens);

/* Free blocks, and the reference count of one block (-1 if out of range). */
PKV_API int32_t pkv_bm_num_free_blocks(const pkv_block_manager* bm);
PKV_API int32_t pkv_bm_refcount(const pkv_block_manager* bm, int32_t block);

/* The free list in order (front first) into out[0 .. *n) if it fits in cap
 * (PKV_EINVAL otherwise, with *n set to the count). */
PKV_API int pkv_bm_free_list(const pkv_block_manager* bm, int32_t* out, int32_t cap, int32_t* n);

/* Pool size from a memory budget (nano-vLLM page, "Implementation du
 * cache"): (usable - model - activation_peak) / bytes of one block over all
 * layers, a block being K and V of block_size tokens, kv_heads heads (those
 * held by this GPU) and d_head elements of dtype_size bytes.  0 when nothing
 * is left; -1 for non-positive shape arguments. */
PKV_API int64_t pkv_blocks_for_budget(int64_t usable_bytes, int64_t model_bytes,
                                      int64_t activation_peak_bytes, int32_t num_layers,
                                      int32_t block_size, int32_t kv_heads, int32_t d_head,
                                      int32_t dtype_size);

/* Device side of copy-on-write: for each i < num_pairs, block pairs[2 i + 1]
 * of both pools becomes a byte copy of block pairs[2 i] (pairs: device int32,
 * as written by pkv_bm_append_tokens).  elem_bytes is 2 for bf16 pools, 1 for
 * FP8 pools; a block is block_size * kv_heads * d_head * elem_bytes bytes and
 * must be a multiple of 16.  No destination may also be a source or appear
 * twice (the copies run concurrently).  Out-of-range ids skip the pair and
 * set PKV_DEVERR_BAD_BLOCK_ID.  This library addition has no counterpart
 * printed in the pages beyond the copy-on-write they name. */
PKV_API int pkv_copy_blocks(void* k_cache, void* v_cache, pkv_cache_desc cache, int32_t elem_bytes,
                            const int32_t* pairs, int32_t num_pairs, pkv_stream_t stream);

#ifdef __cplusplus
}  // extern "C"
#endif

#endif  // PAGEDKV_BLOCKS_H_
