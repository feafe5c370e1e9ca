// Decode attention for callers that cannot allocate device memory.
//
// The split-K decode needs scratch memory for its per-partition partial
// outputs and log-sum-exps.  The regular entry point takes that scratch from
// the caller.  Some callers have no way to provide it: code that runs under a
// fixed, pre-reserved memory budget with no allocator of its own, plug-ins
// that are handed device pointers but may not call cudaMalloc, or serving
// loops that must never allocate (an allocation can synchronise the device or
// fail under memory pressure in the middle of a step).  This entry point
// serves them: it uses a scratch array compiled into the library instead.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes
// (32 MiB).  Every GPU that loads the library holds it until the process
// exits.  Its device address is looked up once per device, on the first call
// made with that device current; make that first call before any stream
// capture.  Nothing in the scratch needs to start at zero: each call writes
// every partial it later reads.  All calls share the one array, so calls
// whose work overlaps on the GPU (different streams, or different host
// threads without ordering) race on it; order them on one stream.
#include <mutex>

#include "../../include/pagedkv.h"
#include "pkv_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up runs on
// the first call per device).  Host code must not use the array's name as a
// device pointer: on the host it only stands in for the symbol.  Only a
// successful lookup is kept: a failed one (e.g. a first call made during a
// stream capture) returns PKV_ECUDA and the next call tries again.
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ECUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();  // leave no sticky launch error behind for the caller
      return PKV_ECUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" {

size_t pkv_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int pkv_paged_decode_attention_noalloc(const void* q, int num_seqs, int q_heads,
                                       const void* k_cache, const void* v_cache,
                                       pkv_cache_desc cache, const int32_t* block_tables,
                                       int max_blocks_per_seq, const int32_t* context_lens,
                                       int max_context_len, float scale, float* out,
                                       int partition_blocks, pkv_stream_t stream) {
  size_t need = 0;
  int st = pkv_decode_plan(num_seqs, q_heads, cache.kv_heads, cache.d_head, max_context_len,
                           partition_blocks, nullptr, nullptr, &need);
  if (st != PKV_OK) return st;
  if (need > kNoAllocScratchBytes) return PKV_ESCRATCH_TOO_SMALL;
  void* scratch = nullptr;
  if (need > 0) {
    st = scratch_for_current_device(&scratch);
    if (st != PKV_OK) return st;
  }
  return pkv_paged_decode_attention_ex(q, num_seqs, q_heads, k_cache, v_cache, cache,
                                       block_tables, max_blocks_per_seq, context_lens,
                                       max_context_len, scale, out, scratch,
                                       need > 0 ? kNoAllocScratchBytes : 0, partition_blocks,
                                       stream);
}

}  // extern "C"
