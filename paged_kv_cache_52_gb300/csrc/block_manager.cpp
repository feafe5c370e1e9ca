// Host block manager of a paged KV cache: a pool of fixed-size blocks handed
// out to sequences, with a first-in first-out free list, reference counts,
// prefix sharing by a chained hash of each full block, and copy-on-write.
//
// The mechanism follows "Maitriser les mecanismes cles de l'inference des
// grands modeles avec nano-vLLM" (section "Implementation du cache": a pool
// allocated at start, a chained hash over the previous block's hash and the
// block's token ids, a reference count protecting shared blocks) and "Cache
// KV, attention et optimisation de l'inference" (sections "PageAtention" and
// "Exercices": 16-token pages anywhere in memory, a free list, copy-on-write
// for a shared system prompt).  The policy choices are listed in the header.
//
// Plain C++ on the host: no CUDA call and no tensor data.
#include <cstdint>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pagedkv_blocks.h"

namespace {

constexpr uint64_t kFnvOffset = 0xcbf29ce484222325ull;
constexpr uint64_t kFnvPrime = 0x100000001b3ull;

// FNV-1a continued from `h` over the little-endian bytes of `n` int32 ids.
uint64_t chain_hash(uint64_t h, const int32_t* ids, int32_t n) {
  for (int32_t i = 0; i < n; ++i) {
    const uint32_t u = static_cast<uint32_t>(ids[i]);
    for (int b = 0; b < 4; ++b) {
      h ^= (u >> (8 * b)) & 0xffu;
      h *= kFnvPrime;
    }
  }
  return h;
}

struct Sequence {
  std::vector<int32_t> blocks;
  std::vector<int32_t> tokens;
  uint64_t last_hash = kFnvOffset;  // hash of the last full block (chain state)
};

}  // namespace

struct pkv_block_manager {
  int32_t num_blocks = 0;
  int32_t bs = 0;
  std::vector<int32_t> ref;
  std::vector<uint64_t> hash;       // cached hash of a full block
  std::vector<uint8_t> hashed;      // 1 if `hash` / `content` are valid
  std::vector<int32_t> content;     // token ids of each hashed block, bs per block
  std::unordered_map<uint64_t, int32_t> by_hash;
  // Free list: doubly linked through prev/next so that a cache hit on a free
  // block leaves the list in O(1); -1 ends it.
  std::vector<int32_t> prev, next;
  std::vector<uint8_t> in_free;
  int32_t head = -1, tail = -1, free_count = 0;
  std::unordered_map<int64_t, Sequence> seqs;

  void push_back_free(int32_t b) {
    prev[b] = tail;
    next[b] = -1;
    if (tail >= 0) next[tail] = b; else head = b;
    tail = b;
    in_free[b] = 1;
    ++free_count;
  }

  void unlink_free(int32_t b) {
    if (prev[b] >= 0) next[prev[b]] = next[b]; else head = next[b];
    if (next[b] >= 0) prev[next[b]] = prev[b]; else tail = prev[b];
    prev[b] = next[b] = -1;
    in_free[b] = 0;
    --free_count;
  }

  // Front of the free list, for new content: its cached hash is dropped.
  int32_t take_free() {
    const int32_t b = head;
    unlink_free(b);
    if (hashed[b]) {
      auto it = by_hash.find(hash[b]);
      if (it != by_hash.end() && it->second == b) by_hash.erase(it);
      hashed[b] = 0;
    }
    ref[b] = 1;
    return b;
  }

  void register_block(int32_t b, uint64_t h, const int32_t* ids) {
    hash[b] = h;
    hashed[b] = 1;
    for (int32_t i = 0; i < bs; ++i) content[size_t(b) * bs + i] = ids[i];
    by_hash[h] = b;
  }

  bool content_equals(int32_t b, const int32_t* ids) const {
    for (int32_t i = 0; i < bs; ++i)
      if (content[size_t(b) * bs + i] != ids[i]) return false;
    return true;
  }

  static int32_t ceil_div(int64_t a, int32_t b) { return int32_t((a + b - 1) / b); }
};

extern "C" {

int pkv_bm_create(int32_t num_blocks, int32_t block_size, pkv_block_manager** out) {
  if (!out) return PKV_EINVAL;
  *out = nullptr;
  if (num_blocks <= 0 || block_size <= 0) return PKV_EINVAL;
  try {
    auto* bm = new pkv_block_manager();
    bm->num_blocks = num_blocks;
    bm->bs = block_size;
    bm->ref.assign(num_blocks, 0);
    bm->hash.assign(num_blocks, 0);
    bm->hashed.assign(num_blocks, 0);
    bm->content.assign(size_t(num_blocks) * block_size, 0);
    bm->prev.assign(num_blocks, -1);
    bm->next.assign(num_blocks, -1);
    bm->in_free.assign(num_blocks, 0);
    for (int32_t b = 0; b < num_blocks; ++b) bm->push_back_free(b);
    *out = bm;
    return PKV_OK;
  } catch (const std::bad_alloc&) {
    return PKV_ENOMEM;
  }
}

void pkv_bm_destroy(pkv_block_manager* bm) { delete bm; }

int pkv_bm_add_sequence(pkv_block_manager* bm, int64_t seq_id, const int32_t* token_ids,
                        int32_t num_tokens, int32_t* num_cached_tokens) {
  if (!bm || num_tokens < 0 || (num_tokens > 0 && !token_ids)) return PKV_EINVAL;
  if (bm->seqs.count(seq_id)) return PKV_EINVAL;
  try {
    const int32_t bs = bm->bs;
    const int32_t nblk = pkv_block_manager::ceil_div(num_tokens, bs);
    const int32_t nfull = num_tokens / bs;
    const int32_t shareable = num_tokens > 0 ? (num_tokens - 1) / bs : 0;
    std::vector<uint64_t> hashes(nfull);
    uint64_t h = kFnvOffset;
    for (int32_t j = 0; j < nfull; ++j) {
      h = chain_hash(h, token_ids + size_t(j) * bs, bs);
      hashes[j] = h;
    }
    std::vector<int32_t> hits;
    for (int32_t j = 0; j < shareable; ++j) {
      auto it = bm->by_hash.find(hashes[j]);
      if (it == bm->by_hash.end() || !bm->content_equals(it->second, token_ids + size_t(j) * bs))
        break;
      hits.push_back(it->second);
    }
    int32_t need = nblk - int32_t(hits.size());
    for (int32_t b : hits) need += bm->ref[b] == 0;
    if (need > bm->free_count) return PKV_ENOBLOCKS;

    Sequence seq;
    seq.blocks.reserve(nblk);
    seq.tokens.assign(token_ids, token_ids + num_tokens);
    seq.last_hash = nfull > 0 ? hashes[nfull - 1] : kFnvOffset;
    for (int32_t b : hits) {
      if (bm->ref[b] == 0) bm->unlink_free(b);
      ++bm->ref[b];
      seq.blocks.push_back(b);
    }
    for (int32_t j = int32_t(hits.size()); j < nblk; ++j) {
      const int32_t b = bm->take_free();
      seq.blocks.push_back(b);
      if (j < nfull) bm->register_block(b, hashes[j], token_ids + size_t(j) * bs);
    }
    bm->seqs.emplace(seq_id, std::move(seq));
    if (num_cached_tokens) *num_cached_tokens = int32_t(hits.size()) * bs;
    return PKV_OK;
  } catch (const std::bad_alloc&) {
    return PKV_ENOMEM;
  }
}

int pkv_bm_append_tokens(pkv_block_manager* bm, int64_t seq_id, const int32_t* token_ids,
                         int32_t num_tokens, int64_t* slots, int32_t* copy_pairs,
                         int32_t max_copies, int32_t* num_copies) {
  if (!bm || num_tokens < 0 || !num_copies) return PKV_EINVAL;
  if (num_tokens > 0 && (!token_ids || !slots)) return PKV_EINVAL;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PKV_EINVAL;
  Sequence& s = it->second;
  const int32_t bs = bm->bs;
  const int64_t L = int64_t(s.tokens.size());
  if (L + num_tokens > INT32_MAX) return PKV_EINVAL;
  const bool cow = num_tokens > 0 && L % bs != 0 && bm->ref[s.blocks.back()] > 1;
  if (cow && (max_copies < 1 || !copy_pairs)) return PKV_EINVAL;
  const int32_t need = int32_t(cow) + pkv_block_manager::ceil_div(L + num_tokens, bs) -
                       pkv_block_manager::ceil_div(L, bs);
  if (need > bm->free_count) return PKV_ENOBLOCKS;
  try {
    s.tokens.reserve(size_t(L + num_tokens));
    s.blocks.reserve(size_t(pkv_block_manager::ceil_div(L + num_tokens, bs)));
  } catch (const std::bad_alloc&) {
    return PKV_ENOMEM;
  }
  *num_copies = 0;
  if (cow) {
    const int32_t old = s.blocks.back();
    const int32_t fresh = bm->take_free();
    --bm->ref[old];
    s.blocks.back() = fresh;
    copy_pairs[0] = old;
    copy_pairs[1] = fresh;
    *num_copies = 1;
  }
  for (int32_t i = 0; i < num_tokens; ++i) {
    const int64_t pos = L + i;
    if (pos % bs == 0) s.blocks.push_back(bm->take_free());
    slots[i] = int64_t(s.blocks[size_t(pos / bs)]) * bs + pos % bs;
  }
  s.tokens.insert(s.tokens.end(), token_ids, token_ids + num_tokens);
  for (int64_t j = L / bs; j < (L + num_tokens) / bs; ++j) {
    const int32_t* chunk = s.tokens.data() + size_t(j) * bs;
    s.last_hash = chain_hash(s.last_hash, chunk, bs);
    bm->register_block(s.blocks[size_t(j)], s.last_hash, chunk);
  }
  return PKV_OK;
}

int pkv_bm_fork(pkv_block_manager* bm, int64_t parent, int64_t child) {
  if (!bm || bm->seqs.count(child)) return PKV_EINVAL;
  auto it = bm->seqs.find(parent);
  if (it == bm->seqs.end()) return PKV_EINVAL;
  try {
    Sequence copy = it->second;
    for (int32_t b : copy.blocks) ++bm->ref[b];
    bm->seqs.emplace(child, std::move(copy));
    return PKV_OK;
  } catch (const std::bad_alloc&) {
    return PKV_ENOMEM;
  }
}

int pkv_bm_free_sequence(pkv_block_manager* bm, int64_t seq_id) {
  if (!bm) return PKV_EINVAL;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PKV_EINVAL;
  const std::vector<int32_t>& blocks = it->second.blocks;
  for (size_t i = blocks.size(); i-- > 0;) {
    const int32_t b = blocks[i];
    if (--bm->ref[b] == 0) bm->push_back_free(b);
  }
  bm->seqs.erase(it);
  return PKV_OK;
}

int pkv_bm_slots(const pkv_block_manager* bm, int64_t seq_id, int32_t start, int32_t count,
                 int64_t* slots) {
  if (!bm || start < 0 || count < 0 || (count > 0 && !slots)) return PKV_EINVAL;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PKV_EINVAL;
  const Sequence& s = it->second;
  if (int64_t(start) + count > int64_t(s.tokens.size())) return PKV_EINVAL;
  for (int32_t i = 0; i < count; ++i) {
    const int64_t pos = int64_t(start) + i;
    slots[i] = int64_t(s.blocks[size_t(pos / bm->bs)]) * bm->bs + pos % bm->bs;
  }
  return PKV_OK;
}

int pkv_bm_seq_len(const pkv_block_manager* bm, int64_t seq_id, int32_t* len) {
  if (!bm || !len) return PKV_EINVAL;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PKV_EINVAL;
  *len = int32_t(it->second.tokens.size());
  return PKV_OK;
}

int pkv_bm_block_table(const pkv_block_manager* bm, int64_t seq_id, int32_t* blocks, int32_t cap,
                       int32_t* num_blocks) {
  if (!bm || !num_blocks) return PKV_EINVAL;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PKV_EINVAL;
  const std::vector<int32_t>& b = it->second.blocks;
  *num_blocks = int32_t(b.size());
  if (int32_t(b.size()) > cap || (!b.empty() && !blocks)) return PKV_EINVAL;
  for (size_t i = 0; i < b.size(); ++i) blocks[i] = b[i];
  return PKV_OK;
}

int pkv_bm_block_tables(const pkv_block_manager* bm, const int64_t* seq_ids, int32_t num_seqs,
                        int32_t* block_tables, int32_t max_blocks_per_seq,
                        int32_t* context_lens) {
  if (!bm || num_seqs < 0 || max_blocks_per_seq < 0) return PKV_EINVAL;
  if (num_seqs == 0) return PKV_OK;
  if (!seq_ids || !context_lens || (max_blocks_per_seq > 0 && !block_tables)) return PKV_EINVAL;
  std::vector<const Sequence*> rows(static_cast<size_t>(num_seqs));
  for (int32_t s = 0; s < num_seqs; ++s) {
    auto it = bm->seqs.find(seq_ids[s]);
    if (it == bm->seqs.end() || int64_t(it->second.blocks.size()) > max_blocks_per_seq)
      return PKV_EINVAL;
    rows[size_t(s)] = &it->second;
  }
  for (int32_t s = 0; s < num_seqs; ++s) {
    const Sequence& q = *rows[size_t(s)];
    int32_t* row = block_tables + size_t(s) * size_t(max_blocks_per_seq);
    for (int32_t j = 0; j < max_blocks_per_seq; ++j)
      row[j] = j < int32_t(q.blocks.size()) ? q.blocks[size_t(j)] : 0;
    context_lens[s] = int32_t(q.tokens.size());
  }
  return PKV_OK;
}

int32_t pkv_bm_num_free_blocks(const pkv_block_manager* bm) { return bm ? bm->free_count : -1; }

int32_t pkv_bm_refcount(const pkv_block_manager* bm, int32_t block) {
  if (!bm || block < 0 || block >= bm->num_blocks) return -1;
  return bm->ref[size_t(block)];
}

int pkv_bm_free_list(const pkv_block_manager* bm, int32_t* out, int32_t cap, int32_t* n) {
  if (!bm || !n) return PKV_EINVAL;
  *n = bm->free_count;
  if (bm->free_count > cap || (bm->free_count > 0 && !out)) return PKV_EINVAL;
  int32_t i = 0;
  for (int32_t b = bm->head; b >= 0; b = bm->next[size_t(b)]) out[i++] = b;
  return PKV_OK;
}

int64_t pkv_blocks_for_budget(int64_t usable_bytes, int64_t model_bytes,
                              int64_t activation_peak_bytes, int32_t num_layers,
                              int32_t block_size, int32_t kv_heads, int32_t d_head,
                              int32_t dtype_size) {
  if (num_layers <= 0 || block_size <= 0 || kv_heads <= 0 || d_head <= 0 || dtype_size <= 0)
    return -1;
  const int64_t per_block = 2 * int64_t(num_layers) * block_size * kv_heads * d_head * dtype_size;
  const int64_t left = usable_bytes - model_bytes - activation_peak_bytes;
  return left > 0 ? left / per_block : 0;
}

}  // extern "C"
