// Chunked-prefill attention over the paged KV cache on the 5th-generation
// tensor cores (tcgen05 + tensor memory).
//
// What is computed ("Optimisation de l'inference", section "Etape 2:
// Attention avec KV Cache"): the n queries of a chunk are the last n positions
// of a sequence whose context (context_len tokens, already appended) lives in
// the paged pools; out = softmax(q K^T * scale + mask) V with the bottom-right
// causal mask (query i of the chunk sees keys 0 .. context_len - n + i), per
// query head, GQA head h reading KV head h / G.  FlashAttention tiling ("Cache
// KV, attention et optimisation de l'inference", "Attention a la lumiere"):
// a 128-row query tile stays on chip while 128-token K/V tiles stream by, with
// a running max and sum.
//
// Design (GB300):
//  * one CTA per (two 128-row query tiles, sequence x KV head).  The 128 rows
//    of a tile are 128/G query tokens x the G heads of the GQA group (rows
//    token-major), so one TMA box brings a tile in and every K/V tile serves
//    all G heads of both tiles.  CTAs are dispatched pair-major: a pair's
//    tiles back to back, longest first (the last tiles of a chunk see the
//    most keys), pairs by context length when an order is given, so the
//    CTAs running together share few pairs' K/V in L2.
//  * warp roles: warps 0-3 and 4-7 are the softmax / correction / epilogue
//    warpgroups of Q tiles 0 and 1 (thread = row = TMEM lane), warp 9 the MMA
//    issuer (one thread), warps 8 and 10 the TMA producers of Q + the K ring
//    (3 stages) and of the V ring (2 stages); their lanes issue the per-page
//    boxes of a 128-key tile.  A K tile is released as soon as both S
//    products have read it, a V tile after both PV products, so each ring
//    refills as early as the MMA order allows.
//  * per Q tile t, tensor memory holds S_t = Q_t K^T (128 fp32 columns) and
//    O_t (d columns).  The softmax overwrites S_t with P_t and the PV product
//    reads P_t straight from tensor memory (A operand in TMEM); V is the
//    MN-major shared-memory operand straight from the pool layout, so no
//    transpose pass and no shared-memory P buffer are needed.
//  * ping-pong: the MMA thread issues PV_0(j), S_0(j+1), PV_1(j), S_1(j+1), so
//    the tensor core works on one tile while the other tile's softmax runs.
//    Consecutive MMAs of the one issuing thread execute in order, which is
//    what lets S_t(j+1) overwrite the P_t(j) that PV_t(j) reads.
//  * P enters the PV product as bf16 hi + bf16 lo (two MMAs per k-step), so
//    its rounding error is ~2^-17 relative instead of bf16's 2^-9 -- needed
//    for rows that see only a few keys, where one rounded weight moves the
//    output by more than 2e-3.
//  * online softmax in base 2 with lazy rescaling: the running max used for
//    the exponentials only moves when a row's new max exceeds it by more than
//    8 (a factor 256), and only then is that row's O rescaled in TMEM.  The
//    final division uses the same stale max for O and the row sum, so the
//    result is exact in real arithmetic.
//  * with P as one f16 operand (F16PV) the row sum adds the weights exactly
//    as they were rounded to f16, so the sum and O weigh every V row alike:
//    the output is a convex combination of V rows whose weights are off by
//    at most 2^-11 relative, and the error reaching it is a weighted mean of
//    those relative errors times (v - out), which vanishes for a row that
//    one key dominates.  The same sum detects a stale max: every weight is
//    at most the tile's sum, so a sum <= 256 proves no weight exceeds 2^8,
//    and after the first tile a CTA takes the exponentials in one pass over
//    the scores with no max pass; only a warp with a larger sum re-reads S
//    (still intact: P is stored last), takes the max and rescales.
//  * every mbarrier wait is bounded; a timeout sets an error bit and an abort
//    flag that the other roles see, copies and MMAs in flight are drained
//    (bounded) and tensor memory is freed before the CTA exits.
#include <algorithm>
#include <climits>

#include "pkv_internal.h"
#include "pkv_prefill_body.cuh"

namespace pkv {

template <int D, int G, bool F16PV, bool PERSIST>
__global__ void __launch_bounds__(kPfThreads, 1)
paged_prefill_kernel(const __grid_constant__ CUtensorMap tmap_q,
                     const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v,
                     const __grid_constant__ CUtensorMap tmap_o, const PrefillParams p) {
  // inputs may have been written by the previous kernel in the stream; with
  // defer_wait the previous kernel wrote nothing this one reads and let it
  // start early, and the wait moves to the end
  if (!p.defer_wait) griddep_wait();
  using L = PrefillSmem<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  volatile int* item_slot = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 8);
  const int warp = threadIdx.x >> 5;
  // tensor memory (warp 0) for the CTA's lifetime
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kPfTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) *abort_flag = 0;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if constexpr (!PERSIST) {
    // grid (pairs, tiles), dispatched in linear block order
    int pair, tile;
    const long long idx = (long long)blockIdx.y * gridDim.x + blockIdx.x;
    if (item_pair_tile(p, idx, int(gridDim.y), pair, tile))
      prefill_item<D, G, F16PV>(tmap_q, tmap_k, tmap_v, tmap_o, p, smem, tmem, pair, tile);
    else if (threadIdx.x == 0)
      atomicOr(&g_prefill_error, kErrBadQueryRange);
  } else {
    // persistent: the same order, taken one item at a time from the counter,
    // so the launch occupies at most gridDim.x SMs
    for (;;) {
      if (threadIdx.x == 0) *item_slot = atomicAdd(p.work_counter, 1);
      __syncthreads();
      const int item = *item_slot;
      const bool stop = item >= p.num_items || *abort_flag;
      __syncthreads();  // every thread has read the slot before it is written again
      if (stop) break;
      int pair, tile;
      if (item_pair_tile(p, item, p.tiles_per_pair, pair, tile))
        prefill_item<D, G, F16PV>(tmap_q, tmap_k, tmap_v, tmap_o, p, smem, tmem, pair, tile);
      else if (threadIdx.x == 0)
        atomicOr(&g_prefill_error, kErrBadQueryRange);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kPfTmemCols);
  }
  if (p.defer_wait) griddep_wait();  // complete only after the previous grid
}

template <int D, int G, bool F16PV>
static cudaError_t launch_prefill_t(const PrefillParams& prm, int max_ctas,
                                    const CUtensorMap* tq, const CUtensorMap* tk,
                                    const CUtensorMap* tv, const CUtensorMap* to,
                                    cudaStream_t stream) {
  using L = PrefillSmem<D>;
  constexpr int TPT = kPfRows / G;
  static std::atomic<int> attr_grid[kAttrMaxDevices], attr_persist[kAttrMaxDevices];
  {
    cudaError_t e =
        set_smem_limit_once(paged_prefill_kernel<D, G, F16PV, false>, L::kSmemBytes, attr_grid);
    if (e == cudaSuccess && F16PV)
      e = set_smem_limit_once(paged_prefill_kernel<D, G, F16PV, F16PV>, L::kSmemBytes,
                              attr_persist);
    if (e != cudaSuccess) return e;
  }
  constexpr int TPC = kPfQTiles * TPT;
  const int tiles = (prm.max_q_len + TPC - 1) / TPC;
  if (prm.work_counter) {
    if (!F16PV) return cudaErrorInvalidValue;  // instantiated for the f16 P V path only
    PrefillParams q = prm;
    const long long items = (long long)prm.num_seqs * prm.kv_heads * tiles;
    if (items > INT32_MAX - 65536) return cudaErrorInvalidValue;
    q.num_items = int(items);
    q.tiles_per_pair = tiles;
    cudaError_t e = cudaMemsetAsync(prm.work_counter, 0, sizeof(int), stream);
    if (e != cudaSuccess) return e;
    const int ctas = int(std::min<long long>(items, max_ctas));
    paged_prefill_kernel<D, G, F16PV, F16PV><<<ctas, kPfThreads, L::kSmemBytes, stream>>>(
        *tq, *tk, *tv, *to, q);
    return cudaGetLastError();
  }
  if (tiles > 65535) return cudaErrorInvalidValue;
  dim3 grid(prm.num_seqs * prm.kv_heads, tiles);
  return launch_after_previous(paged_prefill_kernel<D, G, F16PV, false>, grid, dim3(kPfThreads),
                               L::kSmemBytes, stream, *tq, *tk, *tv, *to, prm);
}

template <int D, bool F16PV>
static cudaError_t launch_prefill_d(const PrefillParams& prm, int max_ctas, int group,
                                    const CUtensorMap* tq, const CUtensorMap* tk,
                                    const CUtensorMap* tv, const CUtensorMap* to,
                                    cudaStream_t st) {
  switch (group) {
    case 1: return launch_prefill_t<D, 1, F16PV>(prm, max_ctas, tq, tk, tv, to, st);
    case 2: return launch_prefill_t<D, 2, F16PV>(prm, max_ctas, tq, tk, tv, to, st);
    case 4: return launch_prefill_t<D, 4, F16PV>(prm, max_ctas, tq, tk, tv, to, st);
    case 8: return launch_prefill_t<D, 8, F16PV>(prm, max_ctas, tq, tk, tv, to, st);
    case 16: return launch_prefill_t<D, 16, F16PV>(prm, max_ctas, tq, tk, tv, to, st);
    default: return cudaErrorInvalidValue;
  }
}

int prefill_rows_per_tile() { return kPfRows; }

cudaError_t launch_paged_prefill(const PrefillArgs& a, const CUtensorMap* tmap_q,
                                 const CUtensorMap* tmap_k, const CUtensorMap* tmap_v,
                                 cudaStream_t stream, const CUtensorMap* tmap_o) {
  PrefillParams prm;
  prm.q_start = a.q_start;
  prm.block_tables = a.block_tables;
  prm.context_lens = a.context_lens;
  prm.out = a.out;
  prm.lse = a.lse;
  prm.context_len = a.context_len;
  prm.out_scale = a.out_scale;
  prm.num_seqs = a.num_seqs;
  prm.q_heads = a.q_heads;
  prm.kv_heads = a.kv_heads;
  prm.num_blocks = a.num_blocks;
  prm.max_blocks_per_seq = a.max_blocks_per_seq;
  prm.total_q = a.total_q;
  prm.max_q_len = a.max_q_len;
  prm.causal = a.causal;
  prm.scale_log2 = a.scale_log2;
  prm.v_block_tables = a.v_block_tables;
  prm.v_num_blocks = a.v_block_tables ? a.v_num_blocks : a.num_blocks;
  prm.work_counter = a.max_ctas > 0 ? a.work_counter : nullptr;
  prm.num_items = 0;        // set by the persistent launch
  prm.tiles_per_pair = 0;
  prm.out_bf16 = a.out_bf16 ? 1 : 0;
  prm.seq_order = a.seq_order;
  prm.table_rows = a.table_rows;
  prm.allow_empty = a.allow_empty ? 1 : 0;
  prm.defer_wait = a.defer_wait ? 1 : 0;
  // without an output map the kernel gets the query map as a stand-in it never uses
  prm.o_tma = (tmap_o && !a.out_bf16) ? 1 : 0;
  const CUtensorMap* to = tmap_o ? tmap_o : tmap_q;
  const int group = a.q_heads / a.kv_heads;
  if (a.f16_pv) {
    if (a.d_head == 128) return launch_prefill_d<128, true>(prm, a.max_ctas, group, tmap_q, tmap_k, tmap_v, to, stream);
    if (a.d_head == 64) return launch_prefill_d<64, true>(prm, a.max_ctas, group, tmap_q, tmap_k, tmap_v, to, stream);
  } else {
    if (a.d_head == 128) return launch_prefill_d<128, false>(prm, a.max_ctas, group, tmap_q, tmap_k, tmap_v, to, stream);
    if (a.d_head == 64) return launch_prefill_d<64, false>(prm, a.max_ctas, group, tmap_q, tmap_k, tmap_v, to, stream);
  }
  return cudaErrorInvalidValue;
}

// Device address of this unit's error word on the current device.
cudaError_t prefill_error_word(unsigned** word) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(word), g_prefill_error);
}

unsigned read_prefill_error(bool clear) {
  unsigned word = 0;
  if (cudaMemcpyFromSymbol(&word, g_prefill_error, sizeof(word)) != cudaSuccess) return ~0u;
  if (clear) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_prefill_error, &zero, sizeof(zero)) != cudaSuccess) return ~0u;
  }
  return word;
}

}  // namespace pkv
