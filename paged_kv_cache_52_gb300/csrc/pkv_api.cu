// C ABI of the paged-KV attention library: argument validation, launch
// planning (split-K partition choice, workspace layout), TMA descriptor
// encoding and error reporting.  All compute runs in the kernels of the other
// translation units; nothing here touches tensor data.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <mutex>

#include "../../include/pagedkv.h"
#include "../../include/pagedkv_blocks.h"
#include "pkv_internal.h"

namespace {

constexpr int kBlockSize = 16;
constexpr int kMaxDevices = 64;

std::atomic<int> g_num_sms[kMaxDevices];

int current_device_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int n = g_num_sms[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_num_sms[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// A library-owned stream per device, with a fork and a join event, for work
// that runs beside a caller's kernel inside one call (the cascade decode's
// prefix pass beside its flat suffix decode).  Created on first use; callers
// hold g_side_mutex from the fork to the join, so the events of two calls
// do not interleave.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
SideStream g_side[kMaxDevices];
std::mutex g_side_mutex;

SideStream* side_stream_locked() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  SideStream& ss = g_side[dev];
  if (!ss.stream) {
    cudaStream_t st = nullptr;
    cudaEvent_t f = nullptr, j = nullptr;
    if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    if (cudaEventCreateWithFlags(&f, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&j, cudaEventDisableTiming) != cudaSuccess) {
      if (f) cudaEventDestroy(f);
      cudaStreamDestroy(st);
      return nullptr;
    }
    ss.stream = st;
    ss.fork = f;
    ss.join = j;
  }
  return &ss;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 4-D view of a pool [num_blocks][16][kv_heads][d_head] bf16, innermost first:
// (d_head, kv_heads, 16, num_blocks).  One box is 64 columns x 1 head x 16
// tokens x 1 block, 128-byte swizzled in shared memory.
bool encode_pool_map(CUtensorMap* map, const void* base, const pkv_cache_desc& c) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[4] = {cuuint64_t(c.d_head), cuuint64_t(c.kv_heads),
                              cuuint64_t(c.block_size), cuuint64_t(c.num_blocks)};
  const cuuint64_t row = cuuint64_t(c.d_head) * 2;
  const cuuint64_t strides[3] = {row, row * cuuint64_t(c.kv_heads),
                                 row * cuuint64_t(c.kv_heads) * cuuint64_t(c.block_size)};
  const cuuint32_t box[4] = {64, 1, cuuint32_t(c.block_size), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D view of packed queries [total_q][q_heads][d_head] bf16: (d_head, q_heads,
// total_q).  One box is 64 columns x `group` heads x `tokens` tokens -- the
// 128 (token, head) rows of one prefill tile, 128-byte swizzled.
bool encode_query_map(CUtensorMap* map, const void* q, int total_q, int q_heads, int d_head,
                      int group, int tokens) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {cuuint64_t(d_head), cuuint64_t(q_heads), cuuint64_t(total_q)};
  const cuuint64_t row = cuuint64_t(d_head) * 2;
  const cuuint64_t strides[2] = {row, row * cuuint64_t(q_heads)};
  const cuuint32_t box[3] = {64, cuuint32_t(group), cuuint32_t(tokens)};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D view of float32 output rows [total_q][q_heads][d_head]: (d_head, q_heads,
// total_q).  One box is 32 columns x `group` heads x 32/group tokens -- the 32
// (token, head) rows one softmax warp of a prefill tile owns -- 128-byte
// swizzled, written by TMA stores.
bool encode_out_map(CUtensorMap* map, void* out, int total_q, int q_heads, int d_head,
                    int group) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc || group <= 0 || group > 32 || 32 % group) return false;
  const cuuint64_t dims[3] = {cuuint64_t(d_head), cuuint64_t(q_heads), cuuint64_t(total_q)};
  const cuuint64_t row = cuuint64_t(d_head) * 4;
  const cuuint64_t strides[2] = {row, row * cuuint64_t(q_heads)};
  const cuuint32_t box[3] = {32, cuuint32_t(group), cuuint32_t(32 / group)};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, out, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// FP8 pool [num_blocks][16][kv_heads][d_head] of e4m3 codes (1 byte): one box
// is a whole 128-byte row x 16 tokens of one head, 128-byte swizzled.
bool encode_pool_map_fp8(CUtensorMap* map, const void* base, const pkv_cache_desc& c) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[4] = {cuuint64_t(c.d_head), cuuint64_t(c.kv_heads),
                              cuuint64_t(c.block_size), cuuint64_t(c.num_blocks)};
  const cuuint64_t row = cuuint64_t(c.d_head);
  const cuuint64_t strides[3] = {row, row * cuuint64_t(c.kv_heads),
                                 row * cuuint64_t(c.kv_heads) * cuuint64_t(c.block_size)};
  const cuuint32_t box[4] = {cuuint32_t(c.d_head), 1, cuuint32_t(c.block_size), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_cache_desc(const pkv_cache_desc& c) {
  if (c.num_blocks <= 0 || c.kv_heads <= 0 || c.d_head <= 0 || c.block_size <= 0)
    return PKV_EINVAL;
  if (c.block_size != kBlockSize) return PKV_EUNSUPPORTED;
  return PKV_OK;
}

bool supported_group(int g) { return g == 1 || g == 2 || g == 4 || g == 8 || g == 16; }

struct Plan {
  int partition_blocks = 1;
  int num_parts = 1;
  size_t ws_bytes = 0;  // covers the uniform plan and, when chosen, the list
  size_t lse_offset = 0;
  // length-balanced work list (bf16 decode only)
  bool list = false;
  int list_target = 0, list_items = 0, list_max_blocks = 0;
  size_t list_lse_offset = 0, list_base_offset = 0;
  // flat split (bf16 decode only): one CTA per SM, partial slots for every
  // pair and every warp, the page prefix sums after them
  bool flat = false;
  int flat_ctas = 0, flat_max_blocks = 0;
  size_t flat_lse_offset = 0, flat_pre_offset = 0;
};

// Partition choice.  Work items are (sequence x KV head, partition).  Long
// partitions amortise each CTA's pipeline start and keep the partial/merge
// traffic small, so the partition is sized for about two items per SM
// (estimated from the longest context).  With more pairs than CTA slots the
// partition is capped at about 150 sqrt(pairs / slots) pages; with fewer,
// it stays within 16..256 pages unless few long contexts fill one wave
// (up to 1024 pages).  The sweeps behind each rule are quoted below.
constexpr int kAutoMinPartBlocks = 16;
constexpr int kAutoMaxPartBlocks = 256;
constexpr int kItemsPerSm = 2;
// The length-balanced list: runs of at least this many pages, and the CTA
// slots of one wave as the run count aimed at.
constexpr int kListMinRun = 8;
// The fused mixed step spreads its prefill items over this share (per mille)
// of its work list; the rest holds decode runs only.  On GB300 the mixed
// step (8 x 512-token chunks + 248 decodes) was fastest with the prefill
// items spread over the whole list: 0.843 ms at 1000, 0.857 at 950, 0.868
// at 900, 0.883 at 800, 0.935 at 500 (with its prefix group; the decode runs
// taking their pages one at a time).
constexpr int kMixedPrefillSpanPermille = 1000;

// Whether the library's own choice (partition_blocks == 0) takes the
// length-balanced list.  Measured on GB300 (70B-GQA recipe, 1 to 64
// sequences) the list never beat the uniform plan: a small batch's time is
// the decode's fixed cost (launch, pipeline ramp, merge) more than the
// balance of its waves.  So the library's choice stays uniform, and the list
// serves PKV_SPLIT_BALANCED, the CTA-capped decode and the fused mixed step.
bool list_wins(long long /*pairs*/, long long /*slots*/) { return false; }

// Whether the library's own choice takes the flat split (d_head 128): for
// 193 to 1024 (sequence, KV head) pairs over bf16 pages (128 to 1024 over
// FP8 pages), and for more pairs when the uniform split needs 3 or more
// partitions per pair, i.e. when the longest context is several times the
// partition the pair count allows, as in a long-tailed batch.  Measured on
// GB300 (decode call, us, uniform / flat): 70B-GQA recipe, 8 sequences 36.2
// / 39.2, 12 44.9 / 44.2, 16 60.5 / 56.2, 24 82.8 / 81.9, 32 120-140 /
// 103.1, 48 160.0 / 146.4, 64 197.4 / 182.5, 96 276.9 / 261.1, 128 353.4 /
// 351.4, 192 535.2 / 535.8, 256 (2 partitions) 696.1 / 704.2; 7B-MHA (2048
// pairs, 1 partition) 368.6 / 376.4; 128K contexts (32 pairs) 320.7 /
// 320.2; the mixed step's 248 decodes (1984 pairs, lognormal contexts up to
// 32768 tokens, 6 partitions) 555.5 / 516.4.  With the uniform split's short
// partitions taking their pages one at a time (bf16): 12 sequences 41.6 /
// 44.9, 16 53.4 / 57.3, 24 81.6 / 81.9, 32 113.5 / 105.1 -- so over bf16
// pages the flat split starts above 24 sequences (192 pairs); the FP8 split
// kernel keeps its pairs and FP8 pools keep the 128-pair start (16
// sequences 42.5 / 39.1).  With fewer pairs a warp's few pages do not
// amortise its start and the pieces' merge; with many pairs in few
// partitions the uniform grid's dynamic CTA scheduling evens out the tail
// that equal static ranges leave.
constexpr long long kFlatMinPairsBf16 = 193;
constexpr long long kFlatMinPairsFp8 = 128;
bool flat_wins(long long pairs, int d_head, long long uniform_parts, bool fp8) {
  if (d_head != 128 || pairs < (fp8 ? kFlatMinPairsFp8 : kFlatMinPairsBf16)) return false;
  return pairs <= 1024 || uniform_parts >= 3;
}

int make_plan(int num_seqs, int q_heads, int kv_heads, int d_head, int max_context_len,
              int partition_blocks, Plan* plan, bool allow_list = false, int list_ctas = 0,
              bool allow_flat = false, bool fp8 = false) {
  *plan = Plan();  // every field is this call's: a plan object may be reused
  if (num_seqs < 0 || q_heads <= 0 || kv_heads <= 0 || max_context_len < 0) return PKV_EINVAL;
  if (q_heads % kv_heads) return PKV_EUNSUPPORTED;
  if (!supported_group(q_heads / kv_heads)) return PKV_EUNSUPPORTED;
  if (d_head != 64 && d_head != 128) return PKV_EUNSUPPORTED;
  if (partition_blocks < PKV_SPLIT_FLAT) return PKV_EINVAL;
  if (partition_blocks == PKV_SPLIT_FLAT && !allow_flat) partition_blocks = PKV_SPLIT_UNIFORM;
  const int max_pb = pkv::decode_max_partition_blocks();
  const int nblk_max = (max_context_len + kBlockSize - 1) / kBlockSize;
  const long long pairs = (long long)num_seqs * kv_heads;
  const int sms = current_device_sms() > 0 ? current_device_sms() : 148;
  const long long slots = (long long)kItemsPerSm * sms;
  int pb;
  if (partition_blocks > 0) {
    if (partition_blocks > max_pb) return PKV_EINVAL;
    pb = partition_blocks;
  } else {
    if (pairs * 4 <= slots && nblk_max >= 4 * kAutoMaxPartBlocks) {
      // Few (sequence, KV head) pairs with long contexts: equal partitions,
      // all in one wave of CTAs (no partly empty last wave), as long as the
      // largest partition allows while every SM still gets a CTA -- a long
      // partition amortises its CTA's pipeline start.  4 x 131072 tokens on
      // GB300: 1024-block partitions (256 CTAs) 0.326 ms, 911 (288 CTAs)
      // 0.335, 256 (1024 CTAs, 3.4 waves) 0.341.
      long long parts = (nblk_max + max_pb - 1) / max_pb;
      const long long floor_parts = (sms + pairs - 1) / pairs;
      if (parts < floor_parts) parts = floor_parts;
      if (parts > slots / pairs) parts = slots / pairs;
      long long want = (nblk_max + parts - 1) / parts;
      if (want > max_pb) want = max_pb;
      pb = int(want);
    } else {
      // about kItemsPerSm work items per SM over the longest context
      long long want = ((long long)nblk_max * pairs + slots - 1) / slots;
      const int lo = nblk_max < kAutoMinPartBlocks ? (nblk_max > 0 ? nblk_max : 1)
                                                   : kAutoMinPartBlocks;
      if (pairs > slots) {
        // More pairs than CTA slots: partitions of about 150 sqrt(pairs /
        // slots) blocks.  Longer ones leave long CTAs for the tail; shorter
        // ones add CTAs, partial rows and merge work.  Measured on GB300 with
        // ragged contexts: 2048 pairs (70B-GQA, 256 sequences) best at 384
        // blocks, 0.699 ms against 0.716 at 256; 1984 pairs (lognormal
        // contexts) 384, 0.554 against 0.562; 512 pairs 192, 0.197 against
        // 0.210.
        const long long cap = (long long)(150.0 * std::sqrt(double(pairs) / double(slots)));
        if (want > cap) want = cap;
        if (want > max_pb) want = max_pb;
      } else if (want > kAutoMaxPartBlocks) {
        want = kAutoMaxPartBlocks;
      }
      if (want < lo) want = lo;
      pb = int(want);
    }
  }
  const long long parts = nblk_max > 0 ? ((long long)nblk_max + pb - 1) / pb : 1;
  if (parts > 65535) return PKV_EUNSUPPORTED;
  plan->partition_blocks = pb;
  plan->num_parts = int(parts);
  if (parts > 1) {
    const size_t rows = size_t(num_seqs) * size_t(q_heads) * size_t(parts);
    const size_t o_bytes = rows * size_t(d_head) * sizeof(float);
    plan->lse_offset = (o_bytes + 255) / 256 * 256;
    plan->ws_bytes = plan->lse_offset + rows * sizeof(float);
  } else {
    plan->ws_bytes = 0;
    plan->lse_offset = 0;
  }
  const bool want_flat = list_ctas == 0 && (partition_blocks == PKV_SPLIT_FLAT ||
                                             (partition_blocks == 0 &&
                                              flat_wins(pairs, d_head, parts, fp8)));
  // the workspace of the library's choice over bf16 pages also serves the
  // FP8 decode of the same sizes, which takes the flat split from fewer pairs
  const bool size_flat =
      want_flat || (list_ctas == 0 && partition_blocks == 0 && flat_wins(pairs, d_head, parts, true));
  if (allow_flat && size_flat) {
    // partial slots for the larger of the bf16 and FP8 flat grids, so one
    // workspace serves both decodes of these sizes
    const long long warps = (long long)sms * std::max(pkv::decode_flat_warps(d_head, false),
                                                      pkv::decode_flat_warps(d_head, true));
    if (num_seqs > pkv::decode_flat_max_seqs() ||
        (long long)sms * pkv::decode_flat_warps(d_head, false) < kv_heads) {
      if (partition_blocks == PKV_SPLIT_FLAT) return PKV_EUNSUPPORTED;
    } else if (num_seqs > 0) {
      // a partial slot for every pair and every warp (at most (S + groups)
      // Hkv pieces; see the flat merge), their log2-sum-exps, then the block
      // prefix sums
      const size_t slots = size_t(pairs + warps) * size_t(q_heads / kv_heads);
      auto up = [](size_t x) { return (x + 255) / 256 * 256; };
      const size_t lse_off = up(slots * size_t(d_head) * sizeof(float));
      const size_t pre_off = lse_off + up(slots * sizeof(float));
      // the workspace still covers the uniform split, which the FP8 and
      // verification decodes take with the same sizes
      plan->ws_bytes = std::max(plan->ws_bytes, pre_off + size_t(num_seqs + 1) * sizeof(int32_t));
      if (want_flat) {
        plan->flat = true;
        plan->flat_ctas = sms;
        plan->flat_max_blocks = nblk_max;
        plan->flat_lse_offset = lse_off;
        plan->flat_pre_offset = pre_off;
        return PKV_OK;
      }
    }
  }
  if (partition_blocks == PKV_SPLIT_FLAT) partition_blocks = PKV_SPLIT_UNIFORM;
  const bool want_list = partition_blocks == PKV_SPLIT_BALANCED || list_ctas > 0 ||
                         (partition_blocks == 0 && list_wins(pairs, slots));
  if (allow_list && want_list && num_seqs > 0 && num_seqs <= pkv::decode_list_max_seqs()) {
    // the run count aimed at: one wave of CTA slots, or, on at most
    // list_ctas CTAs, four runs per CTA (the CTAs take every list_ctas-th
    // run, so short single-run pairs even out)
    const long long target = list_ctas > 0 ? 4LL * list_ctas : slots;
    // runs: at most the target, plus one per pair for the rounding up, plus
    // what the 1024-page cap on a run adds
    const long long cap_runs =
        (pairs * nblk_max + pkv::decode_max_partition_blocks() - 1) /
        pkv::decode_max_partition_blocks();
    const long long items = target + pairs + cap_runs;
    if (items > INT32_MAX / 16) return PKV_EUNSUPPORTED;
    const size_t rows = size_t(items) * size_t(q_heads / kv_heads);
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    plan->list = true;
    plan->list_target = int(target);
    plan->list_items = int(items);
    plan->list_max_blocks = nblk_max;
    plan->list_lse_offset = up(rows * size_t(d_head) * sizeof(float));
    plan->list_base_offset = plan->list_lse_offset + up(rows * sizeof(float));
    const size_t list_bytes = plan->list_base_offset + size_t(num_seqs + 1) * sizeof(int32_t);
    if (list_bytes > plan->ws_bytes) plan->ws_bytes = list_bytes;
  }
  return PKV_OK;
}

// Workspace of the shared-prefix decode: the own pages' partials (always
// written), the prefix part's normalised output and log2-sum-exp, then each
// sequence's first own block and each group's prefix length.  The own pages
// are planned over the whole max_context_len, so a member whose prefix check
// fails (and falls back to its whole context) is still covered.
struct CascadePlan {
  Plan suffix;
  size_t part_o_off = 0, part_lse_off = 0, pre_o_off = 0, pre_lse_off = 0;
  size_t first_off = 0, ctx_off = 0, total = 0;
  size_t flat_pre_off = 0;  // the flat suffix's block prefix sums
};

// SMs the cascade decode leaves to its prefix pass when the suffix takes the
// flat split (a persistent grid that otherwise holds every SM).  The prefix
// pass of the mixed step's 248 decodes (64 tensor-core items of ~20 us)
// takes ~80 us on 16 SMs, well inside the suffix decode, whose HBM-bound
// warps lose nothing on 136 SMs.
constexpr int kCascadePrefixSms = 16;

int make_cascade_plan(int num_seqs, int q_heads, int kv_heads, int d_head, int max_context_len,
                      int num_groups, CascadePlan* cp) {
  if (num_groups < 1) return PKV_EINVAL;
  int st = make_plan(num_seqs, q_heads, kv_heads, d_head, max_context_len, 0, &cp->suffix,
                     /*allow_list=*/false, 0, /*allow_flat=*/true);
  if (st != PKV_OK) return st;
  const int sms = current_device_sms() > 0 ? current_device_sms() : 148;
  if (cp->suffix.flat &&
      (long long)(sms - kCascadePrefixSms) * pkv::decode_flat_warps(d_head) < kv_heads) {
    st = make_plan(num_seqs, q_heads, kv_heads, d_head, max_context_len, 0, &cp->suffix);
    if (st != PKV_OK) return st;
  }
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t rows = size_t(num_seqs) * size_t(q_heads);
  if (cp->suffix.flat) {
    cp->part_o_off = 0;
    cp->part_lse_off = cp->suffix.flat_lse_offset;
    cp->flat_pre_off = cp->suffix.flat_pre_offset;
    cp->pre_o_off = up(cp->suffix.ws_bytes);
  } else {
    const size_t prow = rows * size_t(cp->suffix.num_parts);
    cp->part_o_off = 0;
    cp->part_lse_off = up(prow * d_head * sizeof(float));
    cp->pre_o_off = cp->part_lse_off + up(prow * sizeof(float));
  }
  cp->pre_lse_off = cp->pre_o_off + up(rows * d_head * sizeof(float));
  cp->first_off = cp->pre_lse_off + up(rows * sizeof(float));
  cp->ctx_off = cp->first_off + up(size_t(num_seqs) * sizeof(int32_t));
  cp->total = cp->ctx_off + up(size_t(num_groups) * sizeof(int32_t));
  return PKV_OK;
}

// Argument checks shared by the bf16 and FP8 prefill entry points.
int check_prefill(const void* q, const int32_t* q_start, int num_seqs, int total_q, int max_q_len,
                  int q_heads, const void* k_cache, const void* v_cache,
                  const pkv_cache_desc& cache, const int32_t* block_tables,
                  int max_blocks_per_seq, const int32_t* context_lens, float scale,
                  const void* out) {
  int st = check_cache_desc(cache);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || total_q < 0 || max_q_len < 0 || q_heads <= 0) return PKV_EINVAL;
  if (q_heads % cache.kv_heads) return PKV_EUNSUPPORTED;
  if (!supported_group(q_heads / cache.kv_heads)) return PKV_EUNSUPPORTED;
  if (cache.d_head != 64 && cache.d_head != 128) return PKV_EUNSUPPORTED;
  if (num_seqs == 0 || total_q == 0 || max_q_len == 0) return PKV_OK;
  if (!q || !q_start || !k_cache || !v_cache || !block_tables || !context_lens || !out)
    return PKV_EINVAL;
  if (max_blocks_per_seq <= 0 || !std::isfinite(scale)) return PKV_EINVAL;
  if ((long long)num_seqs * cache.kv_heads > INT32_MAX) return PKV_EUNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(q_start, 4) || !aligned(block_tables, 4) || !aligned(context_lens, 4))
    return PKV_EINVAL;
  return PKV_OK;
}

// Tensor maps and launch of the tensor-core prefill over bf16 K pages.  V is
// a bf16 pool through block_tables, or (f16_pv) an f16 pool of v_num_blocks
// blocks through v_tables (null: block_tables), with P as one f16 operand.
int run_prefill(const void* q, const int32_t* q_start, int num_seqs, int total_q, int max_q_len,
                int q_heads, const void* k_cache, const void* v_cache,
                const pkv_cache_desc& cache, const int32_t* block_tables,
                int max_blocks_per_seq, const int32_t* context_lens, int causal,
                float scale_log2, float out_scale, void* out, cudaStream_t stream,
                bool f16_pv = false, const int32_t* v_tables = nullptr, int v_num_blocks = 0,
                int max_ctas = 0, int* work_counter = nullptr, bool out_bf16 = false,
                const int32_t* seq_order = nullptr) {
  const int group = q_heads / cache.kv_heads;
  const int rows = pkv::prefill_rows_per_tile();
  pkv_cache_desc vdesc = cache;
  if (v_tables) vdesc.num_blocks = v_num_blocks;
  CUtensorMap tq, tk, tv;
  if (!encode_query_map(&tq, q, total_q, q_heads, cache.d_head, group, rows / group) ||
      !encode_pool_map(&tk, k_cache, cache) || !encode_pool_map(&tv, v_cache, vdesc))
    return PKV_ECUDA;
  pkv::PrefillArgs a;
  a.q_start = q_start;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.out = static_cast<float*>(out);
  a.out_bf16 = out_bf16;
  a.num_seqs = num_seqs;
  a.total_q = total_q;
  a.max_q_len = max_q_len;
  a.q_heads = q_heads;
  a.kv_heads = cache.kv_heads;
  a.d_head = cache.d_head;
  a.num_blocks = cache.num_blocks;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.causal = causal ? 1 : 0;
  a.scale_log2 = scale_log2;
  a.out_scale = out_scale;
  a.f16_pv = f16_pv;
  a.v_block_tables = v_tables;
  a.v_num_blocks = v_num_blocks;
  a.max_ctas = max_ctas;
  a.work_counter = work_counter;
  a.seq_order = seq_order;
  // float32 rows leave through TMA stores (bf16 rows through plain stores)
  CUtensorMap to;
  const bool tma_out =
      !out_bf16 && encode_out_map(&to, out, total_q, q_heads, cache.d_head, group);
  cudaError_t e = pkv::launch_paged_prefill(a, &tq, &tk, &tv, stream, tma_out ? &to : nullptr);
  return e == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

// Workspace of the FP8 prefill: bf16 K and V scratch pools of
// num_seqs * max_blocks pages, the scratch block table, the work counter of
// the persistent launch and the sequences' dispatch order (written by the
// page pass).  The bf16 prefill's workspace is the same from v_off on.
struct Fp8PrefillLayout {
  size_t k_off = 0, v_off = 0, table_off = 0, counter_off = 0, order_off = 0, total = 0;
};

bool fp8_prefill_layout(int num_seqs, int max_blocks, int kv_heads, int d_head,
                        Fp8PrefillLayout* w) {
  if (num_seqs <= 0 || max_blocks <= 0 || kv_heads <= 0 || d_head <= 0) return false;
  const long long pages = (long long)num_seqs * max_blocks;
  if (pages > INT32_MAX || (long long)max_blocks * kBlockSize > INT32_MAX) return false;
  const size_t pool = size_t(pages) * kBlockSize * size_t(kv_heads) * size_t(d_head) * 2;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  w->k_off = 0;
  w->v_off = up(pool);
  w->table_off = w->v_off + up(pool);
  w->counter_off = w->table_off + up(size_t(pages) * 4);
  w->order_off = w->counter_off + 256;
  w->total = w->order_off + up(size_t(num_seqs) * 4);
  return true;
}

// Split plan of the multi-query decode: the decode's partitions, with
// num_seqs * q_len rows per query head in the workspace.
int make_verify_plan(int num_seqs, int q_len, int q_heads, int kv_heads, int d_head,
                     int max_context_len, int partition_blocks, Plan* plan) {
  if (q_len <= 0) return PKV_EINVAL;
  int st = make_plan(num_seqs, q_heads, kv_heads, d_head, max_context_len, partition_blocks, plan);
  if (st != PKV_OK) return st;
  if ((long long)(q_heads / kv_heads) * q_len > pkv::verify_max_rows()) return PKV_EUNSUPPORTED;
  if ((long long)num_seqs * q_len > INT32_MAX) return PKV_EUNSUPPORTED;
  if (plan->num_parts > 1) {
    const size_t rows =
        size_t(num_seqs) * size_t(q_len) * size_t(q_heads) * size_t(plan->num_parts);
    plan->lse_offset = (rows * size_t(d_head) * sizeof(float) + 255) / 256 * 256;
    plan->ws_bytes = plan->lse_offset + rows * sizeof(float);
  }
  return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_version(void) { return 100; }

const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "PKV_OK";
    case PKV_EINVAL: return "PKV_EINVAL: invalid argument";
    case PKV_EUNSUPPORTED: return "PKV_EUNSUPPORTED: unsupported shape";
    case PKV_ECUDA: return "PKV_ECUDA: CUDA call or launch failed";
    case PKV_ENOMEM: return "PKV_ENOMEM: workspace too small or host memory exhausted";
    case PKV_EDEVICE_CHECK: return "PKV_EDEVICE_CHECK: device-side check failed";
    case PKV_ETIMEOUT: return "PKV_ETIMEOUT: bounded device wait ran out";
    case PKV_ESCRATCH_TOO_SMALL:
      return "PKV_ESCRATCH_TOO_SMALL: plan needs more than the fixed no-allocation scratch";
    case PKV_ENOBLOCKS: return "PKV_ENOBLOCKS: not enough free KV blocks";
    default: return "unknown pkv status";
  }
}

int pkv_kv_append(const void* k, int64_t k_tok_stride, const void* v, int64_t v_tok_stride,
                  const int64_t* slot_mapping, int64_t num_tokens, void* k_cache,
                  void* v_cache, pkv_cache_desc cache, pkv_stream_t stream) {
  int st = check_cache_desc(cache);
  if (st != PKV_OK) return st;
  if (num_tokens < 0) return PKV_EINVAL;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKV_EINVAL;
  const int64_t row = int64_t(cache.kv_heads) * cache.d_head;
  if (row % 8) return PKV_EUNSUPPORTED;  // rows move as 16-byte vectors
  if (k_tok_stride < row || v_tok_stride < row || k_tok_stride % 8 || v_tok_stride % 8)
    return PKV_EINVAL;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 8))
    return PKV_EINVAL;
  const int sms = current_device_sms();
  if (sms <= 0) return PKV_ECUDA;
  const int64_t num_slots = int64_t(cache.num_blocks) * cache.block_size;
  cudaError_t e = pkv::launch_kv_append(k, k_tok_stride, v, v_tok_stride, slot_mapping,
                                        num_tokens, k_cache, v_cache, num_slots, int(row),
                                        static_cast<cudaStream_t>(stream), sms);
  return e == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

size_t pkv_kv_append_checked_workspace_bytes(pkv_cache_desc cache) {
  if (check_cache_desc(cache) != PKV_OK) return 0;
  const int64_t num_slots = int64_t(cache.num_blocks) * cache.block_size;
  const size_t words = size_t((num_slots + 31) / 32);
  return 256 + (words * 4 + 255) / 256 * 256;  // reject flag, then the slot bitmap
}

int pkv_kv_append_checked(const void* k, int64_t k_tok_stride, const void* v,
                          int64_t v_tok_stride, const int64_t* slot_mapping, int64_t num_tokens,
                          void* k_cache, void* v_cache, pkv_cache_desc cache, void* workspace,
                          size_t ws_bytes, pkv_stream_t stream) {
  int st = check_cache_desc(cache);
  if (st != PKV_OK) return st;
  if (num_tokens < 0) return PKV_EINVAL;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKV_EINVAL;
  const int64_t row = int64_t(cache.kv_heads) * cache.d_head;
  if (row % 8) return PKV_EUNSUPPORTED;
  if (k_tok_stride < row || v_tok_stride < row || k_tok_stride % 8 || v_tok_stride % 8)
    return PKV_EINVAL;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 8))
    return PKV_EINVAL;
  const size_t need = pkv_kv_append_checked_workspace_bytes(cache);
  if (!workspace || ws_bytes < need) return PKV_ENOMEM;
  if (!aligned(workspace, 256)) return PKV_EINVAL;
  const int sms = current_device_sms();
  if (sms <= 0) return PKV_ECUDA;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const int64_t num_slots = int64_t(cache.num_blocks) * cache.block_size;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* reject = reinterpret_cast<int*>(ws);
  unsigned* bitmap = reinterpret_cast<unsigned*>(ws + 256);
  if (cudaMemsetAsync(workspace, 0, need, cs) != cudaSuccess) return PKV_ECUDA;
  cudaError_t e = pkv::launch_slot_duplicates(slot_mapping, num_tokens, num_slots, bitmap, reject,
                                              cs, sms);
  if (e != cudaSuccess) return PKV_ECUDA;
  e = pkv::launch_kv_append(k, k_tok_stride, v, v_tok_stride, slot_mapping, num_tokens, k_cache,
                            v_cache, num_slots, int(row), cs, sms, reject);
  return e == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

int pkv_copy_blocks(void* k_cache, void* v_cache, pkv_cache_desc cache, int32_t elem_bytes,
                    const int32_t* pairs, int32_t num_pairs, pkv_stream_t stream) {
  if (cache.num_blocks <= 0 || cache.block_size <= 0 || cache.kv_heads <= 0 || cache.d_head <= 0)
    return PKV_EINVAL;
  if (elem_bytes != 1 && elem_bytes != 2) return PKV_EINVAL;
  if (num_pairs < 0) return PKV_EINVAL;
  if (num_pairs == 0) return PKV_OK;
  if (!k_cache || !v_cache || !pairs) return PKV_EINVAL;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(pairs, 4)) return PKV_EINVAL;
  const int64_t block_bytes =
      int64_t(cache.block_size) * cache.kv_heads * cache.d_head * elem_bytes;
  if (block_bytes % 16) return PKV_EUNSUPPORTED;
  const int sms = current_device_sms();
  if (sms <= 0) return PKV_ECUDA;
  cudaError_t e = pkv::launch_copy_blocks(k_cache, v_cache, pairs, num_pairs, cache.num_blocks,
                                          block_bytes, static_cast<cudaStream_t>(stream), sms);
  return e == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

int pkv_kv_append_fp8(const void* k, int64_t k_tok_stride, const void* v, int64_t v_tok_stride,
                      const int64_t* slot_mapping, int64_t num_tokens, void* k_cache,
                      void* v_cache, pkv_cache_desc cache, float k_scale, float v_scale,
                      pkv_stream_t stream) {
  int st = check_cache_desc(cache);
  if (st != PKV_OK) return st;
  if (num_tokens < 0) return PKV_EINVAL;
  if (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
    return PKV_EINVAL;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKV_EINVAL;
  const int64_t row = int64_t(cache.kv_heads) * cache.d_head;
  if (row % 16) return PKV_EUNSUPPORTED;  // rows move as 16-code vectors
  if (k_tok_stride < row || v_tok_stride < row || k_tok_stride % 8 || v_tok_stride % 8)
    return PKV_EINVAL;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 8))
    return PKV_EINVAL;
  const int sms = current_device_sms();
  if (sms <= 0) return PKV_ECUDA;
  const float k_inv = 1.0f / k_scale, v_inv = 1.0f / v_scale;
  cudaError_t e = pkv::launch_kv_append_fp8(
      k, k_tok_stride, v, v_tok_stride, slot_mapping, num_tokens, k_cache, v_cache,
      int64_t(cache.num_blocks) * cache.block_size, int(row), k_inv, v_inv,
      static_cast<cudaStream_t>(stream), sms);
  return e == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

int pkv_decode_plan(int num_seqs, int q_heads, int kv_heads, int d_head, int max_context_len,
                    int partition_blocks, int* out_partition_blocks, int* out_num_parts,
                    size_t* out_workspace_bytes) {
  Plan plan;
  const int st = make_plan(num_seqs, q_heads, kv_heads, d_head, max_context_len,
                           partition_blocks, &plan, /*allow_list=*/true, 0, /*allow_flat=*/true);
  if (st != PKV_OK) return st;
  if (out_partition_blocks) *out_partition_blocks = plan.partition_blocks;
  if (out_num_parts) *out_num_parts = plan.num_parts;
  if (out_workspace_bytes) *out_workspace_bytes = plan.ws_bytes;
  return PKV_OK;
}

size_t pkv_decode_workspace_bytes(int num_seqs, int q_heads, int kv_heads, int d_head,
                                  int max_context_len) {
  Plan plan;
  if (make_plan(num_seqs, q_heads, kv_heads, d_head, max_context_len, 0, &plan,
                /*allow_list=*/true, 0, /*allow_flat=*/true) != PKV_OK)
    return 0;
  return plan.ws_bytes;
}

int pkv_decode_plan_uses_list(int num_seqs, int q_heads, int kv_heads, int d_head,
                              int max_context_len, int partition_blocks) {
  Plan plan;
  const int st = make_plan(num_seqs, q_heads, kv_heads, d_head, max_context_len,
                           partition_blocks, &plan, /*allow_list=*/true, 0, /*allow_flat=*/true);
  if (st != PKV_OK) return st;
  return plan.list ? 1 : 0;
}

int pkv_decode_plan_uses_flat(int num_seqs, int q_heads, int kv_heads, int d_head,
                              int max_context_len, int partition_blocks) {
  Plan plan;
  const int st = make_plan(num_seqs, q_heads, kv_heads, d_head, max_context_len,
                           partition_blocks, &plan, /*allow_list=*/true, 0, /*allow_flat=*/true);
  if (st != PKV_OK) return st;
  return plan.flat ? 1 : 0;
}

namespace {

// The bf16-pool decode with a float32 (or, out_bf16, a bf16) output.
int decode_bf16_pool(const void* q, int num_seqs, int q_heads, const void* k_cache,
                     const void* v_cache, pkv_cache_desc cache, const int32_t* block_tables,
                     int max_blocks_per_seq, const int32_t* context_lens, int max_context_len,
                     float scale, void* out, bool out_bf16, void* workspace, size_t ws_bytes,
                     int partition_blocks, pkv_stream_t stream, int list_ctas = 0,
                     const int64_t* step_slots = nullptr) {
  int st = check_cache_desc(cache);
  if (st != PKV_OK) return st;
  Plan plan;
  st = make_plan(num_seqs, q_heads, cache.kv_heads, cache.d_head, max_context_len,
                 partition_blocks, &plan, /*allow_list=*/true, list_ctas, /*allow_flat=*/true);
  if (st != PKV_OK) return st;
  if (list_ctas > 0 && !plan.list) return PKV_EUNSUPPORTED;  // more than 512 sequences
  if (num_seqs == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PKV_EINVAL;
  if (max_blocks_per_seq <= 0) return PKV_EINVAL;
  if (!std::isfinite(scale)) return PKV_EINVAL;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4) ||
      !aligned(out, out_bf16 ? 2 : 4))
    return PKV_EINVAL;
  if (plan.ws_bytes > 0) {
    if (!workspace || ws_bytes < plan.ws_bytes) return PKV_ENOMEM;
    if (!aligned(workspace, 256)) return PKV_EINVAL;
  }
  CUtensorMap tk, tv;
  if (!encode_pool_map(&tk, k_cache, cache) || !encode_pool_map(&tv, v_cache, cache))
    return PKV_ECUDA;
  pkv::DecodeArgs a;
  a.q = q;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.out = static_cast<float*>(out);
  a.out_bf16 = out_bf16;
  a.part_o = plan.ws_bytes ? static_cast<float*>(workspace) : nullptr;
  a.part_lse = plan.ws_bytes ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                        plan.lse_offset)
                             : nullptr;
  a.num_seqs = num_seqs;
  a.q_heads = q_heads;
  a.kv_heads = cache.kv_heads;
  a.d_head = cache.d_head;
  a.num_blocks = cache.num_blocks;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.partition_blocks = plan.partition_blocks;
  a.num_parts = plan.num_parts;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out_scale = 1.f;
  if (plan.list) {
    if (!workspace || ws_bytes < plan.ws_bytes) return PKV_ENOMEM;  // the list's partials
    char* ws = static_cast<char*>(workspace);
    a.list = true;
    a.part_o = reinterpret_cast<float*>(ws);
    a.part_lse = reinterpret_cast<float*>(ws + plan.list_lse_offset);
    a.list_base = reinterpret_cast<int32_t*>(ws + plan.list_base_offset);
    a.list_target = plan.list_target;
    a.list_min_run = kListMinRun;
    a.list_max_blocks = std::min(plan.list_max_blocks, max_blocks_per_seq);
    a.list_items = plan.list_items;
    a.list_max_ctas = list_ctas;
  }
  if (plan.flat) {
    char* ws = static_cast<char*>(workspace);
    a.flat = true;
    a.part_o = reinterpret_cast<float*>(ws);
    a.part_lse = reinterpret_cast<float*>(ws + plan.flat_lse_offset);
    a.flat_pre = reinterpret_cast<int32_t*>(ws + plan.flat_pre_offset);
    a.flat_ctas = plan.flat_ctas;
    a.flat_max_blocks = std::min(plan.flat_max_blocks, max_blocks_per_seq);
  }
  if (step_slots) {  // the decode step: the append just launched runs beside the decode
    if (plan.list) return PKV_EUNSUPPORTED;
    a.wait_late = true;
    a.step_slots = step_slots;
  }
  cudaError_t e = plan.flat
                      ? pkv::launch_paged_decode_flat(a, &tk, &tv, static_cast<cudaStream_t>(stream))
                      : pkv::launch_paged_decode(a, &tk, &tv, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

}  // namespace

int pkv_paged_decode_attention_ex(const void* q, int num_seqs, int q_heads, const void* k_cache,
                                  const void* v_cache, pkv_cache_desc cache,
                                  const int32_t* block_tables, int max_blocks_per_seq,
                                  const int32_t* context_lens, int max_context_len, float scale,
                                  float* out, void* workspace, size_t ws_bytes,
                                  int partition_blocks, pkv_stream_t stream) {
  return decode_bf16_pool(q, num_seqs, q_heads, k_cache, v_cache, cache, block_tables,
                          max_blocks_per_seq, context_lens, max_context_len, scale, out, false,
                          workspace, ws_bytes, partition_blocks, stream);
}

int pkv_paged_decode_step(const void* q, int num_seqs, int q_heads, const void* k_new,
                          int64_t k_tok_stride, const void* v_new, int64_t v_tok_stride,
                          const int64_t* slot_mapping, void* k_cache, void* v_cache,
                          pkv_cache_desc cache, const int32_t* block_tables,
                          int max_blocks_per_seq, const int32_t* context_lens,
                          int max_context_len, float scale, float* out, void* workspace,
                          size_t ws_bytes, pkv_stream_t stream) {
  int st = check_cache_desc(cache);
  if (st != PKV_OK) return st;
  if (num_seqs < 0) return PKV_EINVAL;
  if (num_seqs == 0) return PKV_OK;
  // the append's checks (pkv_kv_append) ...
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return PKV_EINVAL;
  const int64_t row = int64_t(cache.kv_heads) * cache.d_head;
  if (row % 8) return PKV_EUNSUPPORTED;
  if (k_tok_stride < row || v_tok_stride < row || k_tok_stride % 8 || v_tok_stride % 8)
    return PKV_EINVAL;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(slot_mapping, 8)) return PKV_EINVAL;
  // ... and the decode's, before anything is launched
  Plan plan;
  st = make_plan(num_seqs, q_heads, cache.kv_heads, cache.d_head, max_context_len, 0, &plan,
                 /*allow_list=*/true, 0, /*allow_flat=*/true);
  if (st != PKV_OK) return st;
  if (!q || !block_tables || !context_lens || !out || max_blocks_per_seq <= 0 ||
      !std::isfinite(scale))
    return PKV_EINVAL;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4) || !aligned(out, 4))
    return PKV_EINVAL;
  if (plan.ws_bytes > 0 && (!workspace || ws_bytes < plan.ws_bytes)) return PKV_ENOMEM;
  if (plan.ws_bytes > 0 && !aligned(workspace, 256)) return PKV_EINVAL;
  const int sms = current_device_sms();
  if (sms <= 0) return PKV_ECUDA;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e = pkv::launch_kv_append(k_new, k_tok_stride, v_new, v_tok_stride, slot_mapping,
                                        num_seqs, k_cache, v_cache,
                                        int64_t(cache.num_blocks) * cache.block_size, int(row),
                                        cs, sms, nullptr, /*trigger_dependents=*/true);
  if (e != cudaSuccess) return PKV_ECUDA;
  return decode_bf16_pool(q, num_seqs, q_heads, k_cache, v_cache, cache, block_tables,
                          max_blocks_per_seq, context_lens, max_context_len, scale, out, false,
                          workspace, ws_bytes, 0, stream, 0, slot_mapping);
}

size_t pkv_decode_limited_workspace_bytes(int num_seqs, int q_heads, int kv_heads, int d_head,
                                          int max_context_len, int max_ctas) {
  if (max_ctas < 1) return 0;
  Plan plan;
  if (make_plan(num_seqs, q_heads, kv_heads, d_head, max_context_len, PKV_SPLIT_BALANCED, &plan,
                /*allow_list=*/true, max_ctas) != PKV_OK ||
      !plan.list)
    return 0;
  return plan.ws_bytes;
}

int pkv_paged_decode_attention_limited(const void* q, int num_seqs, int q_heads,
                                       const void* k_cache, const void* v_cache,
                                       pkv_cache_desc cache, const int32_t* block_tables,
                                       int max_blocks_per_seq, const int32_t* context_lens,
                                       int max_context_len, float scale, float* out, int max_ctas,
                                       void* workspace, size_t ws_bytes, pkv_stream_t stream) {
  if (max_ctas < 1) return PKV_EINVAL;
  return decode_bf16_pool(q, num_seqs, q_heads, k_cache, v_cache, cache, block_tables,
                          max_blocks_per_seq, context_lens, max_context_len, scale, out, false,
                          workspace, ws_bytes, PKV_SPLIT_BALANCED, stream, max_ctas);
}

namespace {

// Workspace of the fused mixed step: the f16 prefill's part (V pages in f16,
// their table, its counter and dispatch order), then the decode list's
// partials and plan, then the fused launch's counter.
struct MixedLayout {
  Fp8PrefillLayout pre;  // offsets from its v_off
  Plan dec;
  size_t pre_bytes = 0, dec_off = 0, counter_off = 0, total = 0;
  // decode prefix groups: the prefix part's output and log2-sum-exp, each
  // decode's first own block, each group's prefix length
  size_t pre_o_off = 0, pre_lse_off = 0, first_off = 0, ctx_off = 0;
};

int mixed_layout(int num_prefill, int prefill_max_blocks, int num_decode, int q_heads,
                 int kv_heads, int d_head, int max_decode_context_len, int num_groups,
                 MixedLayout* m) {
  if (!fp8_prefill_layout(num_prefill, prefill_max_blocks, kv_heads, d_head, &m->pre))
    return PKV_EUNSUPPORTED;
  const int sms = current_device_sms() > 0 ? current_device_sms() : 148;
  const int st = make_plan(num_decode, q_heads, kv_heads, d_head, max_decode_context_len,
                           PKV_SPLIT_BALANCED, &m->dec, /*allow_list=*/true, 2 * sms);
  if (st != PKV_OK) return st;
  if (!m->dec.list) return PKV_EUNSUPPORTED;  // more than 512 decode sequences
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  m->pre_bytes = m->pre.total - m->pre.v_off;
  m->dec_off = up(m->pre_bytes);
  m->counter_off = m->dec_off + up(m->dec.ws_bytes);
  m->total = m->counter_off + 256;
  if (num_groups > 0) {
    const size_t rows = size_t(num_decode) * size_t(q_heads);
    m->pre_o_off = m->total;
    m->pre_lse_off = m->pre_o_off + up(rows * size_t(d_head) * sizeof(float));
    m->first_off = m->pre_lse_off + up(rows * sizeof(float));
    m->ctx_off = m->first_off + up(size_t(num_decode) * sizeof(int32_t));
    m->total = m->ctx_off + up(size_t(num_groups) * sizeof(int32_t));
  }
  return PKV_OK;
}

}  // namespace

size_t pkv_mixed_step_workspace_bytes(int num_prefill, int prefill_max_blocks, int num_decode,
                                      int q_heads, int kv_heads, int d_head,
                                      int max_decode_context_len) {
  return pkv_mixed_step_groups_workspace_bytes(num_prefill, prefill_max_blocks, num_decode,
                                               q_heads, kv_heads, d_head, max_decode_context_len,
                                               0);
}

size_t pkv_mixed_step_groups_workspace_bytes(int num_prefill, int prefill_max_blocks,
                                             int num_decode, int q_heads, int kv_heads,
                                             int d_head, int max_decode_context_len,
                                             int num_groups) {
  MixedLayout m;
  if (num_groups < 0 ||
      mixed_layout(num_prefill, prefill_max_blocks, num_decode, q_heads, kv_heads, d_head,
                   max_decode_context_len, num_groups, &m) != PKV_OK)
    return 0;
  return m.total;
}

int pkv_mixed_step_attention_ex(const void* q_prefill, const int32_t* q_start, int num_prefill,
                                int total_q, int max_q_len, const int32_t* prefill_block_tables,
                                int prefill_max_blocks, const int32_t* prefill_context_lens,
                                int causal, const void* q_decode, int num_decode,
                                const int32_t* decode_block_tables, int decode_max_blocks,
                                const int32_t* decode_context_lens, int max_decode_context_len,
                                int q_heads, const void* k_cache, const void* v_cache,
                                pkv_cache_desc cache, float scale, float* out_prefill,
                                float* out_decode, const int32_t* decode_group_start,
                                const int32_t* decode_group_prefix_blocks, int num_groups,
                                int max_group_size, int max_prefix_blocks, void* workspace,
                                size_t ws_bytes, int prefill_span_permille, pkv_stream_t stream) {
  if (prefill_span_permille < 0 || prefill_span_permille > 1000) return PKV_EINVAL;
  if (num_groups < 0) return PKV_EINVAL;
  if (num_groups > 0 && (!decode_group_start || !decode_group_prefix_blocks ||
                         !aligned(decode_group_start, 4) ||
                         !aligned(decode_group_prefix_blocks, 4) || max_group_size < 1 ||
                         max_prefix_blocks < 1))
    return PKV_EINVAL;
  if (prefill_span_permille == 0) prefill_span_permille = kMixedPrefillSpanPermille;
  int st = check_prefill(q_prefill, q_start, num_prefill, total_q, max_q_len, q_heads, k_cache,
                         v_cache, cache, prefill_block_tables, prefill_max_blocks,
                         prefill_context_lens, scale, out_prefill);
  if (st != PKV_OK) return st;
  if (num_prefill <= 0 || total_q <= 0 || max_q_len <= 0 || num_decode <= 0)
    return PKV_EINVAL;  // both parts are needed; the separate calls serve one alone
  if (!q_decode || !decode_block_tables || !decode_context_lens || !out_decode ||
      decode_max_blocks <= 0 || max_decode_context_len < 0)
    return PKV_EINVAL;
  if (!aligned(q_decode, 16) || !aligned(decode_block_tables, 4) ||
      !aligned(decode_context_lens, 4) || !aligned(out_decode, 16))
    return PKV_EINVAL;
  MixedLayout m;
  st = mixed_layout(num_prefill, prefill_max_blocks, num_decode, q_heads, cache.kv_heads,
                    cache.d_head, max_decode_context_len, num_groups, &m);
  if (st != PKV_OK) return st;
  if (!workspace || ws_bytes < m.total) return PKV_ENOMEM;
  if (!aligned(workspace, 256)) return PKV_EINVAL;
  const int sms = current_device_sms();
  if (sms <= 0) return PKV_ECUDA;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // 1. the chunks' V pages to f16 (and the sequences ranked by length)
  int32_t* vtab = reinterpret_cast<int32_t*>(ws + (m.pre.table_off - m.pre.v_off));
  int32_t* order = reinterpret_cast<int32_t*>(ws + (m.pre.order_off - m.pre.v_off));
  cudaError_t e = pkv::launch_v_pages_to_f16(
      v_cache, prefill_block_tables, prefill_context_lens, num_prefill, prefill_max_blocks,
      cache.num_blocks, int64_t(kBlockSize) * cache.kv_heads * cache.d_head, ws, vtab, order, cs,
      sms);
  if (e != cudaSuccess) return PKV_ECUDA;
  // 2. tensor maps: prefill queries, the K and V pools, the f16 V scratch
  const int group = q_heads / cache.kv_heads;
  pkv_cache_desc vdesc = cache;
  vdesc.num_blocks = num_prefill * prefill_max_blocks;
  CUtensorMap tq, tk, tv, tv16;
  if (!encode_query_map(&tq, q_prefill, total_q, q_heads, cache.d_head, group,
                        pkv::prefill_rows_per_tile() / group) ||
      !encode_pool_map(&tk, k_cache, cache) || !encode_pool_map(&tv, v_cache, cache) ||
      !encode_pool_map(&tv16, ws, vdesc))
    return PKV_ECUDA;
  pkv::PrefillArgs pa;
  pa.q_start = q_start;
  pa.block_tables = prefill_block_tables;
  pa.context_lens = prefill_context_lens;
  pa.out = out_prefill;
  pa.num_seqs = num_prefill;
  pa.total_q = total_q;
  pa.max_q_len = max_q_len;
  pa.q_heads = q_heads;
  pa.kv_heads = cache.kv_heads;
  pa.d_head = cache.d_head;
  pa.num_blocks = cache.num_blocks;
  pa.max_blocks_per_seq = prefill_max_blocks;
  pa.causal = causal ? 1 : 0;
  pa.scale_log2 = scale * 1.4426950408889634f;
  pa.f16_pv = true;
  pa.v_block_tables = vtab;
  pa.v_num_blocks = vdesc.num_blocks;
  pa.seq_order = order;
  pkv::DecodeArgs da;
  uint8_t* dws = ws + m.dec_off;
  da.q = q_decode;
  da.block_tables = decode_block_tables;
  da.context_lens = decode_context_lens;
  da.out = out_decode;
  da.part_o = reinterpret_cast<float*>(dws);
  da.part_lse = reinterpret_cast<float*>(dws + m.dec.list_lse_offset);
  da.num_seqs = num_decode;
  da.q_heads = q_heads;
  da.kv_heads = cache.kv_heads;
  da.d_head = cache.d_head;
  da.num_blocks = cache.num_blocks;
  da.max_blocks_per_seq = decode_max_blocks;
  da.scale_log2 = scale * 1.4426950408889634f;
  da.out_scale = 1.f;
  da.list = true;
  da.list_base = reinterpret_cast<int32_t*>(dws + m.dec.list_base_offset);
  da.list_target = m.dec.list_target;
  da.list_min_run = kListMinRun;
  da.list_max_blocks = std::min(m.dec.list_max_blocks, decode_max_blocks);
  da.list_items = m.dec.list_items;
  pkv::PrefillArgs qa;  // the prefix groups' pass over the decode queries
  CUtensorMap tqd;
  if (num_groups > 0) {
    float* pre_o = reinterpret_cast<float*>(ws + m.pre_o_off);
    float* pre_lse = reinterpret_cast<float*>(ws + m.pre_lse_off);
    int32_t* seq_first = reinterpret_cast<int32_t*>(ws + m.first_off);
    int32_t* group_ctx = reinterpret_cast<int32_t*>(ws + m.ctx_off);
    e = pkv::launch_prefix_groups_setup(decode_group_start, decode_group_prefix_blocks,
                                        num_groups, 0, num_decode, decode_block_tables,
                                        decode_max_blocks, decode_context_lens,
                                        std::min(max_prefix_blocks, decode_max_blocks), seq_first,
                                        group_ctx, cs);
    if (e != cudaSuccess) return PKV_ECUDA;
    if (!encode_query_map(&tqd, q_decode, num_decode, q_heads, cache.d_head, group,
                          pkv::prefill_rows_per_tile() / group))
      return PKV_ECUDA;
    qa.q_start = decode_group_start;
    qa.block_tables = decode_block_tables;
    qa.table_rows = decode_group_start;
    qa.context_lens = group_ctx;
    qa.out = pre_o;
    qa.lse = pre_lse;
    qa.num_seqs = num_groups;
    qa.total_q = num_decode;
    qa.max_q_len = max_group_size;
    qa.q_heads = q_heads;
    qa.kv_heads = cache.kv_heads;
    qa.d_head = cache.d_head;
    qa.num_blocks = cache.num_blocks;
    qa.max_blocks_per_seq = decode_max_blocks;
    qa.causal = 0;
    qa.scale_log2 = scale * 1.4426950408889634f;
    qa.allow_empty = true;
    da.seq_first_block = seq_first;
    da.force_partials = 1;
    da.extra_o = pre_o;
    da.extra_lse = pre_lse;
  }
  CUtensorMap to;  // the prefill rows leave through TMA stores
  const bool tma_out = encode_out_map(&to, out_prefill, total_q, q_heads, cache.d_head, group);
  e = pkv::launch_mixed_step(pa, da, reinterpret_cast<int*>(ws + m.counter_off), sms,
                             prefill_span_permille, &tq, &tk, &tv16, &tv, cs,
                             num_groups > 0 ? &qa : nullptr, num_groups > 0 ? &tqd : nullptr,
                             tma_out ? &to : nullptr);
  return e == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

int pkv_mixed_step_attention(const void* q_prefill, const int32_t* q_start, int num_prefill,
                             int total_q, int max_q_len, const int32_t* prefill_block_tables,
                             int prefill_max_blocks, const int32_t* prefill_context_lens,
                             int causal, const void* q_decode, int num_decode,
                             const int32_t* decode_block_tables, int decode_max_blocks,
                             const int32_t* decode_context_lens, int max_decode_context_len,
                             int q_heads, const void* k_cache, const void* v_cache,
                             pkv_cache_desc cache, float scale, float* out_prefill,
                             float* out_decode, void* workspace, size_t ws_bytes,
                             pkv_stream_t stream) {
  return pkv_mixed_step_attention_ex(
      q_prefill, q_start, num_prefill, total_q, max_q_len, prefill_block_tables,
      prefill_max_blocks, prefill_context_lens, causal, q_decode, num_decode, decode_block_tables,
      decode_max_blocks, decode_context_lens, max_decode_context_len, q_heads, k_cache, v_cache,
      cache, scale, out_prefill, out_decode, nullptr, nullptr, 0, 0, 0, workspace, ws_bytes, 0,
      stream);
}

int pkv_paged_decode_attention_bf16out(const void* q, int num_seqs, int q_heads,
                                       const void* k_cache, const void* v_cache,
                                       pkv_cache_desc cache, const int32_t* block_tables,
                                       int max_blocks_per_seq, const int32_t* context_lens,
                                       int max_context_len, float scale, void* out,
                                       void* workspace, size_t ws_bytes, int partition_blocks,
                                       pkv_stream_t stream) {
  return decode_bf16_pool(q, num_seqs, q_heads, k_cache, v_cache, cache, block_tables,
                          max_blocks_per_seq, context_lens, max_context_len, scale, out, true,
                          workspace, ws_bytes, partition_blocks, stream);
}

namespace {

// The FP8-pool decode with a float32 (or, out_bf16, a bf16) output.
int decode_fp8_pool(const void* q, int num_seqs, int q_heads, const void* k_cache,
                    const void* v_cache, pkv_cache_desc cache, const int32_t* block_tables,
                    int max_blocks_per_seq, const int32_t* context_lens, int max_context_len,
                    float scale, float k_scale, float v_scale, void* out, bool out_bf16,
                    void* workspace, size_t ws_bytes, int partition_blocks, pkv_stream_t stream) {
  int st = check_cache_desc(cache);
  if (st != PKV_OK) return st;
  if (cache.d_head != 128) return PKV_EUNSUPPORTED;
  Plan plan;
  st = make_plan(num_seqs, q_heads, cache.kv_heads, cache.d_head, max_context_len,
                 partition_blocks, &plan, /*allow_list=*/false, 0, /*allow_flat=*/true,
                 /*fp8=*/true);
  if (st != PKV_OK) return st;
  if (num_seqs == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PKV_EINVAL;
  if (max_blocks_per_seq <= 0) return PKV_EINVAL;
  if (!std::isfinite(scale) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
    return PKV_EINVAL;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4) ||
      !aligned(out, out_bf16 ? 2 : 4))
    return PKV_EINVAL;
  if (plan.ws_bytes > 0) {
    if (!workspace || ws_bytes < plan.ws_bytes) return PKV_ENOMEM;
    if (!aligned(workspace, 256)) return PKV_EINVAL;
  }
  CUtensorMap tk, tv;
  if (!encode_pool_map_fp8(&tk, k_cache, cache) || !encode_pool_map_fp8(&tv, v_cache, cache))
    return PKV_ECUDA;
  pkv::DecodeArgs a;
  a.q = q;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.out = static_cast<float*>(out);
  a.out_bf16 = out_bf16;
  a.part_o = plan.ws_bytes ? static_cast<float*>(workspace) : nullptr;
  a.part_lse = plan.ws_bytes ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                        plan.lse_offset)
                             : nullptr;
  a.num_seqs = num_seqs;
  a.q_heads = q_heads;
  a.kv_heads = cache.kv_heads;
  a.d_head = cache.d_head;
  a.num_blocks = cache.num_blocks;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.partition_blocks = plan.partition_blocks;
  a.num_parts = plan.num_parts;
  a.scale_log2 = scale * k_scale * 1.4426950408889634f;
  a.out_scale = v_scale;
  if (plan.flat) {
    if ((long long)plan.flat_ctas * pkv::decode_flat_warps(128, true) < cache.kv_heads)
      return PKV_EUNSUPPORTED;
    char* ws = static_cast<char*>(workspace);
    a.flat = true;
    a.fp8 = true;
    a.part_o = reinterpret_cast<float*>(ws);
    a.part_lse = reinterpret_cast<float*>(ws + plan.flat_lse_offset);
    a.flat_pre = reinterpret_cast<int32_t*>(ws + plan.flat_pre_offset);
    a.flat_ctas = plan.flat_ctas;
    a.flat_max_blocks = std::min(plan.flat_max_blocks, max_blocks_per_seq);
    const cudaError_t ef =
        pkv::launch_paged_decode_flat(a, &tk, &tv, static_cast<cudaStream_t>(stream));
    return ef == cudaSuccess ? PKV_OK : PKV_ECUDA;
  }
  cudaError_t e = pkv::launch_paged_decode_fp8(a, &tk, &tv, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

}  // namespace

int pkv_paged_decode_attention_fp8(const void* q, int num_seqs, int q_heads,
                                   const void* k_cache, const void* v_cache, pkv_cache_desc cache,
                                   const int32_t* block_tables, int max_blocks_per_seq,
                                   const int32_t* context_lens, int max_context_len, float scale,
                                   float k_scale, float v_scale, float* out, void* workspace,
                                   size_t ws_bytes, int partition_blocks, pkv_stream_t stream) {
  return decode_fp8_pool(q, num_seqs, q_heads, k_cache, v_cache, cache, block_tables,
                         max_blocks_per_seq, context_lens, max_context_len, scale, k_scale,
                         v_scale, out, false, workspace, ws_bytes, partition_blocks, stream);
}

int pkv_paged_decode_attention_fp8_bf16out(const void* q, int num_seqs, int q_heads,
                                           const void* k_cache, const void* v_cache,
                                           pkv_cache_desc cache, const int32_t* block_tables,
                                           int max_blocks_per_seq, const int32_t* context_lens,
                                           int max_context_len, float scale, float k_scale,
                                           float v_scale, void* out, void* workspace,
                                           size_t ws_bytes, int partition_blocks,
                                           pkv_stream_t stream) {
  return decode_fp8_pool(q, num_seqs, q_heads, k_cache, v_cache, cache, block_tables,
                         max_blocks_per_seq, context_lens, max_context_len, scale, k_scale,
                         v_scale, out, true, workspace, ws_bytes, partition_blocks, stream);
}

int pkv_paged_decode_attention(const void* q, int num_seqs, int q_heads, const void* k_cache,
                               const void* v_cache, pkv_cache_desc cache,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* context_lens, int max_context_len, float scale,
                               float* out, void* workspace, size_t ws_bytes,
                               pkv_stream_t stream) {
  return pkv_paged_decode_attention_ex(q, num_seqs, q_heads, k_cache, v_cache, cache,
                                       block_tables, max_blocks_per_seq, context_lens,
                                       max_context_len, scale, out, workspace, ws_bytes, 0,
                                       stream);
}

int pkv_paged_prefill_attention(const void* q, const int32_t* q_start, int num_seqs, int total_q,
                                int max_q_len, int q_heads, const void* k_cache,
                                const void* v_cache, pkv_cache_desc cache,
                                const int32_t* block_tables, int max_blocks_per_seq,
                                const int32_t* context_lens, int causal, float scale, float* out,
                                pkv_stream_t stream) {
  int st = check_prefill(q, q_start, num_seqs, total_q, max_q_len, q_heads, k_cache, v_cache,
                         cache, block_tables, max_blocks_per_seq, context_lens, scale, out);
  if (st != PKV_OK || num_seqs == 0 || total_q == 0 || max_q_len == 0) return st;
  return run_prefill(q, q_start, num_seqs, total_q, max_q_len, q_heads, k_cache, v_cache, cache,
                     block_tables, max_blocks_per_seq, context_lens, causal,
                     scale * 1.4426950408889634f, 1.f, out, static_cast<cudaStream_t>(stream));
}

size_t pkv_paged_prefill_attention_fp8_workspace_bytes(int num_seqs, int max_blocks_per_seq,
                                                       int kv_heads, int d_head) {
  Fp8PrefillLayout w;
  return fp8_prefill_layout(num_seqs, max_blocks_per_seq, kv_heads, d_head, &w) ? w.total : 0;
}

namespace {

int prefill_fp8(const void* q, const int32_t* q_start, int num_seqs, int total_q, int max_q_len,
                int q_heads, const void* k_cache, const void* v_cache, pkv_cache_desc cache,
                const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                int causal, float scale, float k_scale, float v_scale, float* out,
                void* workspace, size_t ws_bytes, int max_ctas, pkv_stream_t stream) {
  int st = check_prefill(q, q_start, num_seqs, total_q, max_q_len, q_heads, k_cache, v_cache,
                         cache, block_tables, max_blocks_per_seq, context_lens, scale, out);
  if (st != PKV_OK) return st;
  if (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
    return PKV_EINVAL;
  if (num_seqs == 0 || total_q == 0 || max_q_len == 0) return PKV_OK;
  Fp8PrefillLayout w;
  if (!fp8_prefill_layout(num_seqs, max_blocks_per_seq, cache.kv_heads, cache.d_head, &w))
    return PKV_EUNSUPPORTED;
  if (!workspace || ws_bytes < w.total) return PKV_ENOMEM;
  if (!aligned(workspace, 256)) return PKV_EINVAL;
  const int sms = current_device_sms();
  if (sms <= 0) return PKV_ECUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e = pkv::launch_widen_fp8_pages(
      k_cache, v_cache, block_tables, context_lens, num_seqs, max_blocks_per_seq,
      cache.num_blocks, int64_t(kBlockSize) * cache.kv_heads * cache.d_head, ws + w.k_off,
      ws + w.v_off, reinterpret_cast<int32_t*>(ws + w.table_off), /*v_f16=*/true,
      reinterpret_cast<int32_t*>(ws + w.order_off), cs, sms);
  if (e != cudaSuccess) return PKV_ECUDA;
  pkv_cache_desc scratch = cache;
  scratch.num_blocks = num_seqs * max_blocks_per_seq;
  return run_prefill(q, q_start, num_seqs, total_q, max_q_len, q_heads, ws + w.k_off,
                     ws + w.v_off, scratch, reinterpret_cast<const int32_t*>(ws + w.table_off),
                     max_blocks_per_seq, context_lens, causal,
                     scale * k_scale * 1.4426950408889634f, v_scale, out, cs, /*f16_pv=*/true,
                     nullptr, 0, max_ctas, reinterpret_cast<int*>(ws + w.counter_off), false,
                     reinterpret_cast<const int32_t*>(ws + w.order_off));
}

}  // namespace

int pkv_paged_prefill_attention_fp8(const void* q, const int32_t* q_start, int num_seqs,
                                    int total_q, int max_q_len, int q_heads, const void* k_cache,
                                    const void* v_cache, pkv_cache_desc cache,
                                    const int32_t* block_tables, int max_blocks_per_seq,
                                    const int32_t* context_lens, int causal, float scale,
                                    float k_scale, float v_scale, float* out, void* workspace,
                                    size_t ws_bytes, pkv_stream_t stream) {
  return prefill_fp8(q, q_start, num_seqs, total_q, max_q_len, q_heads, k_cache, v_cache, cache,
                     block_tables, max_blocks_per_seq, context_lens, causal, scale, k_scale,
                     v_scale, out, workspace, ws_bytes, 0, stream);
}

int pkv_paged_prefill_attention_fp8_limited(const void* q, const int32_t* q_start, int num_seqs,
                                            int total_q, int max_q_len, int q_heads,
                                            const void* k_cache, const void* v_cache,
                                            pkv_cache_desc cache, const int32_t* block_tables,
                                            int max_blocks_per_seq, const int32_t* context_lens,
                                            int causal, float scale, float k_scale, float v_scale,
                                            float* out, int max_ctas, void* workspace,
                                            size_t ws_bytes, pkv_stream_t stream) {
  if (max_ctas < 1) return PKV_EINVAL;
  return prefill_fp8(q, q_start, num_seqs, total_q, max_q_len, q_heads, k_cache, v_cache, cache,
                     block_tables, max_blocks_per_seq, context_lens, causal, scale, k_scale,
                     v_scale, out, workspace, ws_bytes, max_ctas, stream);
}

size_t pkv_paged_prefill_workspace_bytes(int num_seqs, int max_blocks_per_seq, int kv_heads,
                                         int d_head) {
  Fp8PrefillLayout w;
  if (!fp8_prefill_layout(num_seqs, max_blocks_per_seq, kv_heads, d_head, &w)) return 0;
  return w.total - w.v_off;  // the f16 V pool and the table, no K copy
}

namespace {

int prefill_f16pv(const void* q, const int32_t* q_start, int num_seqs, int total_q,
                  int max_q_len, int q_heads, const void* k_cache, const void* v_cache,
                  pkv_cache_desc cache, const int32_t* block_tables, int max_blocks_per_seq,
                  const int32_t* context_lens, int causal, float scale, void* out,
                  void* workspace, size_t ws_bytes, int max_ctas, pkv_stream_t stream,
                  bool out_bf16 = false) {
  int st = check_prefill(q, q_start, num_seqs, total_q, max_q_len, q_heads, k_cache, v_cache,
                         cache, block_tables, max_blocks_per_seq, context_lens, scale, out);
  if (st != PKV_OK || num_seqs == 0 || total_q == 0 || max_q_len == 0) return st;
  Fp8PrefillLayout w;
  if (!fp8_prefill_layout(num_seqs, max_blocks_per_seq, cache.kv_heads, cache.d_head, &w))
    return PKV_EUNSUPPORTED;
  if (ws_bytes < w.total - w.v_off) return PKV_ENOMEM;
  if (!aligned(workspace, 256)) return PKV_EINVAL;
  const int sms = current_device_sms();
  if (sms <= 0) return PKV_ECUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* vtab = reinterpret_cast<int32_t*>(ws + (w.table_off - w.v_off));
  int32_t* order = reinterpret_cast<int32_t*>(ws + (w.order_off - w.v_off));
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e = pkv::launch_v_pages_to_f16(
      v_cache, block_tables, context_lens, num_seqs, max_blocks_per_seq, cache.num_blocks,
      int64_t(kBlockSize) * cache.kv_heads * cache.d_head, ws, vtab, order, cs, sms);
  if (e != cudaSuccess) return PKV_ECUDA;
  return run_prefill(q, q_start, num_seqs, total_q, max_q_len, q_heads, k_cache, ws, cache,
                     block_tables, max_blocks_per_seq, context_lens, causal,
                     scale * 1.4426950408889634f, 1.f, out, cs, /*f16_pv=*/true, vtab,
                     num_seqs * max_blocks_per_seq, max_ctas,
                     reinterpret_cast<int*>(ws + (w.counter_off - w.v_off)), out_bf16, order);
}

}  // namespace

int pkv_paged_prefill_attention_ex(const void* q, const int32_t* q_start, int num_seqs,
                                   int total_q, int max_q_len, int q_heads, const void* k_cache,
                                   const void* v_cache, pkv_cache_desc cache,
                                   const int32_t* block_tables, int max_blocks_per_seq,
                                   const int32_t* context_lens, int causal, float scale,
                                   float* out, void* workspace, size_t ws_bytes,
                                   pkv_stream_t stream) {
  if (!workspace)
    return pkv_paged_prefill_attention(q, q_start, num_seqs, total_q, max_q_len, q_heads,
                                       k_cache, v_cache, cache, block_tables,
                                       max_blocks_per_seq, context_lens, causal, scale, out,
                                       stream);
  return prefill_f16pv(q, q_start, num_seqs, total_q, max_q_len, q_heads, k_cache, v_cache,
                       cache, block_tables, max_blocks_per_seq, context_lens, causal, scale, out,
                       workspace, ws_bytes, 0, stream);
}

int pkv_paged_prefill_attention_limited(const void* q, const int32_t* q_start, int num_seqs,
                                        int total_q, int max_q_len, int q_heads,
                                        const void* k_cache, const void* v_cache,
                                        pkv_cache_desc cache, const int32_t* block_tables,
                                        int max_blocks_per_seq, const int32_t* context_lens,
                                        int causal, float scale, float* out, int max_ctas,
                                        void* workspace, size_t ws_bytes, pkv_stream_t stream) {
  if (max_ctas < 1) return PKV_EINVAL;
  if (!workspace) return PKV_ENOMEM;
  return prefill_f16pv(q, q_start, num_seqs, total_q, max_q_len, q_heads, k_cache, v_cache,
                       cache, block_tables, max_blocks_per_seq, context_lens, causal, scale, out,
                       workspace, ws_bytes, max_ctas, stream);
}

int pkv_paged_prefill_attention_bf16out(const void* q, const int32_t* q_start, int num_seqs,
                                       int total_q, int max_q_len, int q_heads,
                                       const void* k_cache, const void* v_cache,
                                       pkv_cache_desc cache, const int32_t* block_tables,
                                       int max_blocks_per_seq, const int32_t* context_lens,
                                       int causal, float scale, void* out, void* workspace,
                                       size_t ws_bytes, pkv_stream_t stream) {
  if (workspace)
    return prefill_f16pv(q, q_start, num_seqs, total_q, max_q_len, q_heads, k_cache, v_cache,
                         cache, block_tables, max_blocks_per_seq, context_lens, causal, scale,
                         out, workspace, ws_bytes, 0, stream, /*out_bf16=*/true);
  int st = check_prefill(q, q_start, num_seqs, total_q, max_q_len, q_heads, k_cache, v_cache,
                         cache, block_tables, max_blocks_per_seq, context_lens, scale, out);
  if (st != PKV_OK || num_seqs == 0 || total_q == 0 || max_q_len == 0) return st;
  return run_prefill(q, q_start, num_seqs, total_q, max_q_len, q_heads, k_cache, v_cache, cache,
                     block_tables, max_blocks_per_seq, context_lens, causal,
                     scale * 1.4426950408889634f, 1.f, out, static_cast<cudaStream_t>(stream),
                     false, nullptr, 0, 0, nullptr, /*out_bf16=*/true);
}

size_t pkv_verify_workspace_bytes(int num_seqs, int q_len, int q_heads, int kv_heads, int d_head,
                                  int max_context_len, int partition_blocks) {
  Plan plan;
  if (make_verify_plan(num_seqs, q_len, q_heads, kv_heads, d_head, max_context_len,
                       partition_blocks, &plan) != PKV_OK)
    return 0;
  return plan.ws_bytes;
}

namespace {

// The multi-query decode with a float32 (or, out_bf16, a bf16) output.
int verify_bf16_pool(const void* q, int num_seqs, int q_len, int q_heads, const void* k_cache,
                     const void* v_cache, pkv_cache_desc cache, const int32_t* block_tables,
                     int max_blocks_per_seq, const int32_t* context_lens, int max_context_len,
                     float scale, void* out, bool out_bf16, void* workspace, size_t ws_bytes,
                     int partition_blocks, pkv_stream_t stream) {
  int st = check_cache_desc(cache);
  if (st != PKV_OK) return st;
  Plan plan;
  st = make_verify_plan(num_seqs, q_len, q_heads, cache.kv_heads, cache.d_head, max_context_len,
                        partition_blocks, &plan);
  if (st != PKV_OK) return st;
  if (num_seqs == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PKV_EINVAL;
  if (max_blocks_per_seq <= 0 || !std::isfinite(scale)) return PKV_EINVAL;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4) ||
      !aligned(out, out_bf16 ? 2 : 4))
    return PKV_EINVAL;
  if (plan.ws_bytes > 0) {
    if (!workspace || ws_bytes < plan.ws_bytes) return PKV_ENOMEM;
    if (!aligned(workspace, 256)) return PKV_EINVAL;
  }
  CUtensorMap tk, tv;
  if (!encode_pool_map(&tk, k_cache, cache) || !encode_pool_map(&tv, v_cache, cache))
    return PKV_ECUDA;
  pkv::DecodeArgs a;
  a.q = q;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.out = static_cast<float*>(out);
  a.out_bf16 = out_bf16;
  a.part_o = plan.ws_bytes ? static_cast<float*>(workspace) : nullptr;
  a.part_lse = plan.ws_bytes ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                        plan.lse_offset)
                             : nullptr;
  a.num_seqs = num_seqs;
  a.q_heads = q_heads;
  a.kv_heads = cache.kv_heads;
  a.d_head = cache.d_head;
  a.num_blocks = cache.num_blocks;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.partition_blocks = plan.partition_blocks;
  a.num_parts = plan.num_parts;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out_scale = 1.f;
  cudaError_t e = pkv::launch_paged_verify(a, q_len, &tk, &tv, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

}  // namespace

int pkv_paged_verify_attention(const void* q, int num_seqs, int q_len, int q_heads,
                               const void* k_cache, const void* v_cache, pkv_cache_desc cache,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* context_lens, int max_context_len, float scale,
                               float* out, void* workspace, size_t ws_bytes,
                               int partition_blocks, pkv_stream_t stream) {
  return verify_bf16_pool(q, num_seqs, q_len, q_heads, k_cache, v_cache, cache, block_tables,
                          max_blocks_per_seq, context_lens, max_context_len, scale, out, false,
                          workspace, ws_bytes, partition_blocks, stream);
}

int pkv_paged_verify_attention_bf16out(const void* q, int num_seqs, int q_len, int q_heads,
                                       const void* k_cache, const void* v_cache,
                                       pkv_cache_desc cache, const int32_t* block_tables,
                                       int max_blocks_per_seq, const int32_t* context_lens,
                                       int max_context_len, float scale, void* out,
                                       void* workspace, size_t ws_bytes, int partition_blocks,
                                       pkv_stream_t stream) {
  return verify_bf16_pool(q, num_seqs, q_len, q_heads, k_cache, v_cache, cache, block_tables,
                          max_blocks_per_seq, context_lens, max_context_len, scale, out, true,
                          workspace, ws_bytes, partition_blocks, stream);
}

size_t pkv_decode_shared_prefix_workspace_bytes(int num_seqs, int q_heads, int kv_heads,
                                                 int d_head, int max_context_len,
                                                 int prefix_blocks) {
  if (prefix_blocks <= 0) return 0;
  CascadePlan cp;
  if (make_cascade_plan(num_seqs, q_heads, kv_heads, d_head, max_context_len, 1, &cp) != PKV_OK)
    return 0;
  return cp.total;
}

size_t pkv_decode_prefix_groups_workspace_bytes(int num_seqs, int q_heads, int kv_heads,
                                                int d_head, int max_context_len,
                                                int num_groups) {
  CascadePlan cp;
  if (make_cascade_plan(num_seqs, q_heads, kv_heads, d_head, max_context_len, num_groups, &cp) !=
      PKV_OK)
    return 0;
  return cp.total;
}

}  // extern "C"

namespace {

// The shared-prefix (cascade) decode over prefix groups.  group_start null:
// one group of all sequences with uniform_prefix_blocks.
int cascade_decode(const void* q, int num_seqs, int q_heads, const void* k_cache,
                   const void* v_cache, pkv_cache_desc cache, const int32_t* block_tables,
                   int max_blocks_per_seq, const int32_t* context_lens, int max_context_len,
                   const int32_t* group_start, const int32_t* group_prefix_blocks,
                   int num_groups, int max_group_size, int max_prefix_blocks,
                   int uniform_prefix_blocks, float scale, float* out, void* workspace,
                   size_t ws_bytes, pkv_stream_t stream) {
  int st = check_cache_desc(cache);
  if (st != PKV_OK) return st;
  const bool uniform = group_start == nullptr;
  const int groups = uniform ? 1 : num_groups;
  if (groups < 1 || max_prefix_blocks < 1 || max_group_size < 1) return PKV_EINVAL;
  CascadePlan cp;
  st = make_cascade_plan(num_seqs, q_heads, cache.kv_heads, cache.d_head, max_context_len, groups,
                         &cp);
  if (st != PKV_OK) return st;
  if (num_seqs == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PKV_EINVAL;
  if (!uniform && !group_prefix_blocks) return PKV_EINVAL;
  if (max_blocks_per_seq < 1 || !std::isfinite(scale)) return PKV_EINVAL;
  if ((long long)num_seqs > 65535 * 128LL) return PKV_EUNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4) || !aligned(out, 4) ||
      (!uniform && (!aligned(group_start, 4) || !aligned(group_prefix_blocks, 4))))
    return PKV_EINVAL;
  if (!workspace || ws_bytes < cp.total) return PKV_ENOMEM;
  if (!aligned(workspace, 256)) return PKV_EINVAL;
  char* ws = static_cast<char*>(workspace);
  float* pre_o = reinterpret_cast<float*>(ws + cp.pre_o_off);
  float* pre_lse = reinterpret_cast<float*>(ws + cp.pre_lse_off);
  int32_t* seq_first = reinterpret_cast<int32_t*>(ws + cp.first_off);
  int32_t* group_ctx = reinterpret_cast<int32_t*>(ws + cp.ctx_off);
  const int group = q_heads / cache.kv_heads;
  const float scale_log2 = scale * 1.4426950408889634f;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // 0. each sequence's first own block (its members checked against the
  //    group leader's ids) and each group's prefix length
  cudaError_t e = pkv::launch_prefix_groups_setup(
      group_start, group_prefix_blocks, num_groups, uniform_prefix_blocks, num_seqs, block_tables,
      max_blocks_per_seq, context_lens, std::min(max_prefix_blocks, max_blocks_per_seq), seq_first,
      group_ctx, s);
  if (e != cudaSuccess) return PKV_ECUDA;

  CUtensorMap tq, tk, tv;
  const int rows_per_tile = pkv::prefill_rows_per_tile();
  if (!encode_query_map(&tq, q, num_seqs, q_heads, cache.d_head, group, rows_per_tile / group) ||
      !encode_pool_map(&tk, k_cache, cache) || !encode_pool_map(&tv, v_cache, cache))
    return PKV_ECUDA;

  // 1. the decode of each sequence's own blocks after its prefix, partials
  //    only
  pkv::DecodeArgs a;
  a.q = q;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.out = out;
  a.part_o = reinterpret_cast<float*>(ws + cp.part_o_off);
  a.part_lse = reinterpret_cast<float*>(ws + cp.part_lse_off);
  a.num_seqs = num_seqs;
  a.q_heads = q_heads;
  a.kv_heads = cache.kv_heads;
  a.d_head = cache.d_head;
  a.num_blocks = cache.num_blocks;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.partition_blocks = cp.suffix.partition_blocks;
  a.num_parts = cp.suffix.num_parts;
  a.scale_log2 = scale_log2;
  a.out_scale = 1.f;
  a.seq_first_block = seq_first;
  a.force_partials = 1;
  a.extra_o = pre_o;
  a.extra_lse = pre_lse;
  a.early_trigger = true;
  a.skip_merge = true;

  // 2. the prefix pass: every group's queries against its prefix keys,
  //    non-causal, on the tensor cores (a group is one pseudo-sequence of its
  //    members' rows)
  pkv::PrefillArgs pa;
  pa.q_start = group_start;       // null: one group of all rows
  pa.block_tables = block_tables;
  pa.table_rows = group_start;    // a group reads its leader's row (null: row 0)
  pa.context_lens = group_ctx;
  pa.out = pre_o;
  pa.lse = pre_lse;
  pa.num_seqs = groups;
  pa.total_q = num_seqs;
  pa.max_q_len = uniform ? num_seqs : max_group_size;
  pa.q_heads = q_heads;
  pa.kv_heads = cache.kv_heads;
  pa.d_head = cache.d_head;
  pa.num_blocks = cache.num_blocks;
  pa.max_blocks_per_seq = max_blocks_per_seq;
  pa.causal = 0;
  pa.scale_log2 = scale_log2;
  pa.allow_empty = true;          // a group with an invalid prefix has none

  if (cp.suffix.flat) {
    // 1'-2'. the own blocks on the flat split, on all but kCascadePrefixSms
    //    SMs, and the prefix pass beside it on the library's side stream
    //    (forked after the setup, joined before the merge): the flat grid
    //    holds its SMs to the end, so the prefix pass gets SMs of its own
    a.flat = true;
    a.flat_pre = reinterpret_cast<int32_t*>(ws + cp.flat_pre_off);
    a.flat_ctas = current_device_sms() - kCascadePrefixSms;
    a.flat_max_blocks = std::min(cp.suffix.flat_max_blocks, max_blocks_per_seq);
    a.early_trigger = false;
    if (a.flat_ctas < 1) return PKV_ECUDA;
    std::lock_guard<std::mutex> lock(g_side_mutex);
    SideStream* side = side_stream_locked();
    if (!side) return PKV_ECUDA;
    if (cudaEventRecord(side->fork, s) != cudaSuccess) return PKV_ECUDA;
    e = pkv::launch_paged_decode_flat(a, &tk, &tv, s);
    if (e != cudaSuccess) return PKV_ECUDA;
    if (cudaStreamWaitEvent(side->stream, side->fork, 0) != cudaSuccess) return PKV_ECUDA;
    pa.defer_wait = false;
    e = pkv::launch_paged_prefill(pa, &tq, &tk, &tv, side->stream);
    if (e != cudaSuccess) return PKV_ECUDA;
    if (cudaEventRecord(side->join, side->stream) != cudaSuccess ||
        cudaStreamWaitEvent(s, side->join, 0) != cudaSuccess)
      return PKV_ECUDA;
    // 3'. the merge folds the prefix part in as one more piece
    e = pkv::launch_paged_decode_flat_merge(a, s);
    return e == cudaSuccess ? PKV_OK : PKV_ECUDA;
  }

  // 1-2. the uniform split, whose CTAs let the next launch start while they
  //    run, then the prefix pass: it fills the SMs the decode's last CTAs
  //    leave, and waits for the decode only before it finishes
  e = pkv::launch_paged_decode(a, &tk, &tv, s);
  if (e != cudaSuccess) return PKV_ECUDA;
  pa.defer_wait = true;
  e = pkv::launch_paged_prefill(pa, &tq, &tk, &tv, s);
  if (e != cudaSuccess) return PKV_ECUDA;

  // 3. the merge folds the prefix part in as one more partial
  e = pkv::launch_paged_decode_merge_only(a, s);
  return e == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

}  // namespace

extern "C" {

int pkv_paged_decode_attention_shared_prefix(
    const void* q, int num_seqs, int q_heads, const void* k_cache, const void* v_cache,
    pkv_cache_desc cache, const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* context_lens, int max_context_len, int prefix_blocks, float scale, float* out,
    void* workspace, size_t ws_bytes, pkv_stream_t stream) {
  if (prefix_blocks <= 0 || prefix_blocks > max_blocks_per_seq) return PKV_EINVAL;
  return cascade_decode(q, num_seqs, q_heads, k_cache, v_cache, cache, block_tables,
                        max_blocks_per_seq, context_lens, max_context_len, nullptr, nullptr, 1,
                        num_seqs > 0 ? num_seqs : 1, prefix_blocks, prefix_blocks, scale, out,
                        workspace, ws_bytes, stream);
}

int pkv_paged_decode_attention_prefix_groups(
    const void* q, int num_seqs, int q_heads, const void* k_cache, const void* v_cache,
    pkv_cache_desc cache, const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* context_lens, int max_context_len, const int32_t* group_start,
    const int32_t* group_prefix_blocks, int num_groups, int max_group_size,
    int max_prefix_blocks, float scale, float* out, void* workspace, size_t ws_bytes,
    pkv_stream_t stream) {
  if (!group_start) return PKV_EINVAL;
  return cascade_decode(q, num_seqs, q_heads, k_cache, v_cache, cache, block_tables,
                        max_blocks_per_seq, context_lens, max_context_len, group_start,
                        group_prefix_blocks, num_groups, max_group_size, max_prefix_blocks, 0,
                        scale, out, workspace, ws_bytes, stream);
}

}  // extern "C"

namespace {

// The error words of every kernel unit, gathered on a stream: one thread
// reads each word -- and, with `clear`, exchanges it for 0 in the same
// atomic step, so a bit raised meanwhile by a kernel on another stream stays
// for the next query instead of being lost -- and stores the OR.
struct ErrorWordSet {
  unsigned* word[9];
  int count;
  int clear;
};

__device__ unsigned g_collected_error = 0;

__global__ void collect_error_words_kernel(const ErrorWordSet s) {
  unsigned acc = 0;
  for (int i = 0; i < s.count; ++i)
    acc |= s.clear ? atomicExch(s.word[i], 0u) : atomicOr(s.word[i], 0u);
  g_collected_error = acc;
}

std::mutex g_collect_mutex;  // one collection in flight per process

int collect_error_words(cudaStream_t stream, bool clear, unsigned* word) {
  ErrorWordSet s = {};
  cudaError_t (*const getters[9])(unsigned**) = {
      pkv::append_error_word, pkv::decode_error_word, pkv::decode_fp8_error_word,
      pkv::prefill_error_word, pkv::verify_error_word, pkv::probe_error_word,
      pkv::mixed_decode_error_word, pkv::mixed_prefill_error_word, pkv::decode_flat_error_word};
  for (int i = 0; i < 9; ++i)
    if (getters[i](&s.word[i]) != cudaSuccess) return PKV_ECUDA;
  s.count = 9;
  s.clear = clear ? 1 : 0;
  std::lock_guard<std::mutex> lock(g_collect_mutex);
  collect_error_words_kernel<<<1, 1, 0, stream>>>(s);
  if (cudaGetLastError() != cudaSuccess) return PKV_ECUDA;
  unsigned w = 0;
  if (cudaMemcpyFromSymbolAsync(&w, g_collected_error, sizeof(w), 0, cudaMemcpyDeviceToHost,
                                stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return PKV_ECUDA;
  *word = w;
  return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_get_last_device_error_bits(pkv_stream_t stream, unsigned int* word) {
  unsigned w = 0;
  const int st = collect_error_words(static_cast<cudaStream_t>(stream), true, &w);
  if (st != PKV_OK) return st;
  if (word) *word = w;
  if (w & PKV_DEVERR_WAIT_TIMEOUT) return PKV_ETIMEOUT;
  return w ? PKV_EDEVICE_CHECK : PKV_OK;
}

int pkv_get_last_device_error(pkv_stream_t stream) {
  return pkv_get_last_device_error_bits(stream, nullptr);
}

int pkv_get_device_error(unsigned int* word, int clear) {
  if (!word) return PKV_EINVAL;
  if (cudaDeviceSynchronize() != cudaSuccess) return PKV_ECUDA;
  const unsigned a = pkv::read_append_error(clear != 0);
  const unsigned d = pkv::read_decode_error(clear != 0);
  const unsigned f = pkv::read_prefill_error(clear != 0);
  const unsigned d8 = pkv::read_decode_fp8_error(clear != 0);
  const unsigned v = pkv::read_verify_error(clear != 0);
  const unsigned w = pkv::read_probe_error(clear != 0);
  const unsigned m = pkv::read_mixed_error(clear != 0);
  const unsigned fl = pkv::read_decode_flat_error(clear != 0);
  if (a == ~0u || d == ~0u || f == ~0u || d8 == ~0u || v == ~0u || w == ~0u || m == ~0u ||
      fl == ~0u)
    return PKV_ECUDA;
  *word = a | d | f | d8 | v | w | m | fl;
  return PKV_OK;
}

uint32_t pkv_wait_poll_limit(void) { return pkv::wait_poll_limit(); }

int pkv_wait_timeout_probe(uint32_t polls, unsigned long long* cycles, pkv_stream_t stream) {
  if (polls == 0 || polls > pkv::wait_poll_limit()) return PKV_EINVAL;
  if (cycles && !aligned(cycles, 8)) return PKV_EINVAL;
  const cudaError_t e =
      pkv::launch_wait_timeout_probe(polls, cycles, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

}  // extern "C"
