// The continuous-batching step's attention as one persistent launch: the
// chunked-prefill query tiles (tensor cores) and the decode runs (HBM) are
// items of one work list, taken by every SM from one counter.
//
// What is computed ("第 10 讲：推理（Inference）", "核心概念与定义":
// continuous batching, selective batching -- attention per sequence; the
// nano-vLLM page, section "Priorité au pré-remplissage"): the outputs of the
// chunked prefill of the new prompts and of the decode step of the running
// sequences, exactly as pkv_paged_prefill_attention_ex and the length-balanced
// list decode give them.
//
// Design (GB300):
//  * one CTA per SM (the prefill item needs 225 KB of shared memory and all
//    512 tensor-memory columns), 11 warps.  A CTA takes list positions from a
//    counter; a position is either a prefill item (two 128-row query tiles of
//    one sequence x KV head, computed with the prefill kernel's warp roles) or
//    a decode run (pages of one sequence x KV head, computed by the warps
//    whose 3-stage TMA rings fit below the prefill's bookkeeping -- 9 at
//    d_head 128 (216 KB in flight), 8 at 64 -- each as in the decode kernel).
//  * the prefill items are spread evenly over the list (or over its first
//    part, a parameter), so at any moment the CTAs share out between
//    tensor-bound prefill items and HBM-bound decode runs in proportion to
//    the work left of each kind, and both kinds finish together.
//  * the decode runs come from the list plan (a one-CTA plan kernel before
//    this launch); runs of one pair are merged afterwards by the list merge.
//  * with prefix groups (decodes whose first pages are the same physical
//    blocks), the list starts with the groups' prefix items: each group's
//    member queries attend its prefix once on the tensor cores, and the
//    decode runs cover only each member's own pages; the merge folds the
//    prefix part in.
//  * every mbarrier wait is bounded; a prefill item that times out raises the
//    abort flag, and the CTA stops taking items.
#include "pkv_decode_body.cuh"
#include "pkv_internal.h"
#include "pkv_prefill_body.cuh"

namespace pkv {

// Warps that own decode rings in a mixed CTA: as many 3-stage rings as fit
// below the prefill's bookkeeping (9 at d_head 128, 8 at 64).
template <int D>
struct MixedDecodeWarps {
  static constexpr int value = DecodeTile<D, 9>::kEnd <= PrefillSmem<D>::kMiscOff ? 9 : 8;
};

struct MixedParams {
  int* counter;                  // list positions taken, zeroed by the plan kernel
  const int32_t* seq_item_base;  // the decode plan ([num_decode + 1]), written by the plan kernel
  int num_prefill_items;         // prefill pairs x tiles_per_pair
  int tiles_per_pair;
  int prefill_span_permille;     // the prefill items are spread over this share of the list
  // decode prefix groups: the first num_prefix_items positions attend each
  // group's shared prefix for its members' queries (0: no groups)
  int num_prefix_items;          // groups x KV heads x prefix_tiles
  int prefix_tiles;
};

template <int D>
struct MixedSmem {
  static constexpr int kPrefill = PrefillSmem<D>::kSmemBytes;
  static constexpr int kDecode = DecodeTile<D, MixedDecodeWarps<D>::value>::kSmemBytes;
  static constexpr int kSmemBytes = kPrefill > kDecode ? kPrefill : kDecode;
  static_assert(kSmemBytes <= 232448, "mixed-step CTA does not fit in shared memory");
  // the prefill's own bookkeeping (tensor-memory address, abort flag, item
  // slot) lies past every decode buffer
  static_assert(PrefillSmem<D>::kMiscOff >= DecodeTile<D, MixedDecodeWarps<D>::value>::kEnd,
                "decode buffers overlap the prefill's bookkeeping");
};

// The decode list plan for the mixed step (one CTA), and the zeroed counter.
__global__ void __launch_bounds__(512) mixed_plan_kernel(const DecodeParams p,
                                                        const DecodeListParams lp, int* counter) {
  griddep_wait();
  list_plan<512>(p, lp, lp.seq_item_base);
  if (threadIdx.x == 0) *counter = 0;
}

template <int D, int G>
__global__ void __launch_bounds__(kPfThreads, 1)
paged_mixed_step_kernel(const __grid_constant__ CUtensorMap tmap_q,
                        const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v16,
                        const __grid_constant__ CUtensorMap tmap_v,
                        const __grid_constant__ CUtensorMap tmap_qd,
                        const __grid_constant__ CUtensorMap tmap_o, const PrefillParams pp,
                        const PrefillParams pq, const DecodeParams dp, const DecodeListParams lp,
                        const MixedParams mp) {
  griddep_wait();  // the plan, the f16 V pages and the appended rows are in place
  using L = PrefillSmem<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  volatile int* item_slot = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kPfTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) *abort_flag = 0;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const long long Q = mp.num_prefix_items;
  const long long P = mp.num_prefill_items;
  const long long rest = P + mp.seq_item_base[lp.num_seqs];
  long long span = rest * mp.prefill_span_permille / 1000;
  if (span < P) span = P;
  if (span < 1) span = 1;
  for (;;) {
    if (threadIdx.x == 0) *item_slot = atomicAdd(mp.counter, 1);
    __syncthreads();
    const long long at = *item_slot;
    const bool stop = at >= Q + rest || *abort_flag;
    __syncthreads();  // every thread has read the slot before it is written again
    if (stop) break;
    if (at < Q) {
      // a prefix-group item: the members' queries against the group's prefix
      // (bf16 V from the pool, P as hi + lo), writing the extra partial
      const int per_group = pq.kv_heads * mp.prefix_tiles;
      const int grp = int(at / per_group);
      const int r = int(at - (long long)grp * per_group);
      const int kvh = r / mp.prefix_tiles;
      const int tile = mp.prefix_tiles - 1 - (r - kvh * mp.prefix_tiles);
      // (the prefix partials are written row by row: tmap_qd only fills the
      // output map's place)
      prefill_item<D, G, false>(tmap_qd, tmap_k, tmap_v, tmap_qd, pq, smem, tmem,
                                grp * pq.kv_heads + kvh, tile);
      fence_proxy_async_smem();
      __syncthreads();
      continue;
    }
    const long long pos = at - Q;
    // prefill items before position pos: floor(pos P / span) inside the span
    const long long before = pos < span ? pos * P / span : P;
    const bool is_prefill = pos < span && (pos + 1) * P / span > before;
    if (is_prefill) {
      int pair, tile;
      if (item_pair_tile(pp, before, mp.tiles_per_pair, pair, tile))
        prefill_item<D, G, true>(tmap_q, tmap_k, tmap_v16, tmap_o, pp, smem, tmem, pair, tile);
      else if (threadIdx.x == 0)
        atomicOr(&g_prefill_error, kErrBadQueryRange);
    } else {
      // one page at a time: beside the prefill items' traffic these runs are
      // bound by the bytes each warp keeps in flight, and refilling a stage
      // as soon as its page is done keeps more in flight than pairs
      list_item<D, G, MixedDecodeWarps<D>::value, false>(tmap_k, tmap_v, dp, lp, smem,
                                                          mp.seq_item_base, int(pos - before));
      __syncthreads();  // every warp has left the run's merge
      // the run's barriers are retired: this memory holds prefill tiles next
      if (warp < MixedDecodeWarps<D>::value && lane == 0)
        for (int st = 0; st < kDecodeStages; ++st)
          mbar_inval(smem_u32(smem + DecodeTile<D, MixedDecodeWarps<D>::value>::kBarOffset) +
                     (warp * kDecodeStages + st) * 8);
    }
    // the item's generic shared-memory accesses come before the next item's
    // copies into the same memory
    fence_proxy_async_smem();
    __syncthreads();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kPfTmemCols);
  }
}

struct MixedLaunch {
  const CUtensorMap *tmap_q, *tmap_k, *tmap_v16, *tmap_v, *tmap_qd, *tmap_o;
  const PrefillParams* pp;
  const PrefillParams* pq;
  const DecodeParams* dp;
  const DecodeListParams* lp;
  const MixedParams* mp;
  int ctas;
};

template <int D, int G>
static cudaError_t launch_mixed_t(const MixedLaunch& m, cudaStream_t stream) {
  using S = MixedSmem<D>;
  static std::atomic<int> attr_done[kAttrMaxDevices];
  cudaError_t e = set_smem_limit_once(paged_mixed_step_kernel<D, G>, S::kSmemBytes, attr_done);
  if (e != cudaSuccess) return e;
  return launch_after_previous(paged_mixed_step_kernel<D, G>, dim3(unsigned(m.ctas)),
                               dim3(kPfThreads), S::kSmemBytes, stream, *m.tmap_q, *m.tmap_k,
                               *m.tmap_v16, *m.tmap_v, *m.tmap_qd, *m.tmap_o, *m.pp, *m.pq,
                               *m.dp, *m.lp, *m.mp);
}

template <int D>
static cudaError_t launch_mixed_d(const MixedLaunch& m, int group, cudaStream_t st) {
  switch (group) {
    case 1: return launch_mixed_t<D, 1>(m, st);
    case 2: return launch_mixed_t<D, 2>(m, st);
    case 4: return launch_mixed_t<D, 4>(m, st);
    case 8: return launch_mixed_t<D, 8>(m, st);
    case 16: return launch_mixed_t<D, 16>(m, st);
    default: return cudaErrorInvalidValue;
  }
}

static PrefillParams prefill_params(const PrefillArgs& a) {
  PrefillParams pp;
  pp.q_start = a.q_start;
  pp.block_tables = a.block_tables;
  pp.context_lens = a.context_lens;
  pp.out = a.out;
  pp.lse = a.lse;
  pp.context_len = 0;
  pp.out_scale = 1.f;
  pp.num_seqs = a.num_seqs;
  pp.q_heads = a.q_heads;
  pp.kv_heads = a.kv_heads;
  pp.num_blocks = a.num_blocks;
  pp.max_blocks_per_seq = a.max_blocks_per_seq;
  pp.total_q = a.total_q;
  pp.max_q_len = a.max_q_len;
  pp.causal = a.causal;
  pp.scale_log2 = a.scale_log2;
  pp.v_block_tables = a.v_block_tables;
  pp.v_num_blocks = a.v_block_tables ? a.v_num_blocks : a.num_blocks;
  pp.work_counter = nullptr;
  pp.num_items = 0;
  pp.tiles_per_pair = 0;
  pp.out_bf16 = 0;
  pp.seq_order = a.seq_order;
  pp.table_rows = a.table_rows;
  pp.allow_empty = a.allow_empty ? 1 : 0;
  pp.defer_wait = 0;
  return pp;
}

cudaError_t launch_mixed_step(const PrefillArgs& pa, const DecodeArgs& da, int* counter,
                              int ctas, int prefill_span_permille, const CUtensorMap* tmap_q,
                              const CUtensorMap* tmap_k, const CUtensorMap* tmap_v16,
                              const CUtensorMap* tmap_v, cudaStream_t stream,
                              const PrefillArgs* prefix, const CUtensorMap* tmap_qd,
                              const CUtensorMap* tmap_o) {
  // prefill part: the f16 P V path over the f16 V scratch pages
  PrefillParams pp = prefill_params(pa);
  pp.o_tma = tmap_o ? 1 : 0;
  constexpr int TPC = kPfQTiles * kPfRows;  // query rows per item
  const int group = pa.q_heads / pa.kv_heads;
  const int tokens_per_item = TPC / group;
  const int tiles = pa.num_seqs > 0 ? (pa.max_q_len + tokens_per_item - 1) / tokens_per_item : 0;
  const long long items = (long long)pa.num_seqs * pa.kv_heads * tiles;
  if (items > INT32_MAX / 2) return cudaErrorInvalidValue;
  pp.num_items = int(items);
  pp.tiles_per_pair = tiles;
  // decode part: the list plan's runs
  DecodeParams dp;
  dp.q = static_cast<const __nv_bfloat16*>(da.q);
  dp.block_tables = da.block_tables;
  dp.context_lens = da.context_lens;
  dp.out = da.out;
  dp.part_o = da.part_o;
  dp.part_lse = da.part_lse;
  dp.q_heads = da.q_heads;
  dp.kv_heads = da.kv_heads;
  dp.num_blocks = da.num_blocks;
  dp.max_blocks_per_seq = da.max_blocks_per_seq;
  dp.partition_blocks = 1;
  dp.num_parts = 1;
  dp.scale_log2 = da.scale_log2;
  dp.out_scale = 1.f;
  dp.first_block = 0;
  dp.force_partials = 0;
  dp.extra_o = nullptr;
  dp.extra_lse = nullptr;
  dp.out_bf16 = 0;
  dp.seq_first_block = da.seq_first_block;
  dp.force_partials = da.force_partials;
  dp.extra_o = da.extra_o;
  dp.extra_lse = da.extra_lse;
  // prefix-group items (none without groups)
  PrefillParams pq = prefix ? prefill_params(*prefix) : pp;
  long long qitems = 0;
  int qtiles = 0;
  if (prefix) {
    qtiles = (prefix->max_q_len + tokens_per_item - 1) / tokens_per_item;
    qitems = (long long)prefix->num_seqs * prefix->kv_heads * qtiles;
    if (qitems > INT32_MAX / 2) return cudaErrorInvalidValue;
  }
  DecodeListParams lp;
  lp.seq_item_base = da.list_base;
  lp.num_seqs = da.num_seqs;
  lp.target_items = da.list_target;
  lp.min_run = da.list_min_run;
  lp.max_blocks = da.list_max_blocks;
  MixedParams mp;
  mp.counter = counter;
  mp.seq_item_base = da.list_base;
  mp.num_prefill_items = int(items);
  mp.tiles_per_pair = tiles;
  mp.prefill_span_permille = prefill_span_permille;
  mp.num_prefix_items = int(qitems);
  mp.prefix_tiles = qtiles;
  // 1. the decode plan (and the zeroed counter)
  cudaError_t e = launch_after_previous(mixed_plan_kernel, dim3(1), dim3(512), 0, stream, dp, lp,
                                        counter);
  if (e != cudaSuccess) return e;
  // 2. the fused launch
  MixedLaunch m{tmap_q, tmap_k, tmap_v16, tmap_v, prefix ? tmap_qd : tmap_q,
                tmap_o ? tmap_o : tmap_q, &pp, &pq, &dp, &lp, &mp, ctas};
  if (pa.d_head == 128) e = launch_mixed_d<128>(m, group, stream);
  else if (pa.d_head == 64) e = launch_mixed_d<64>(m, group, stream);
  else e = cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  // 3. the runs of each decode pair merged
  return launch_decode_list_merge(dp, lp, pa.d_head, stream);
}

// Device addresses of this unit's error words (its copies of the decode and
// prefill bodies' words) on the current device.
cudaError_t mixed_decode_error_word(unsigned** word) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(word), g_decode_error);
}
cudaError_t mixed_prefill_error_word(unsigned** word) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(word), g_prefill_error);
}

unsigned read_mixed_error(bool clear) {
  unsigned a = 0, b = 0;
  if (cudaMemcpyFromSymbol(&a, g_decode_error, sizeof(a)) != cudaSuccess ||
      cudaMemcpyFromSymbol(&b, g_prefill_error, sizeof(b)) != cudaSuccess)
    return ~0u;
  if (clear) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_decode_error, &zero, sizeof(zero)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_prefill_error, &zero, sizeof(zero)) != cudaSuccess)
      return ~0u;
  }
  return a | b;
}

}  // namespace pkv
