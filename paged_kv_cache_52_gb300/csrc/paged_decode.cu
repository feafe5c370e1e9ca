// Paged decode attention with split-K (flash-decoding) and a log-sum-exp
// merge.
//
// What is computed ("Optimisation de l'inference", section "Etape 2:
// Attention avec KV Cache"; "Cache KV, attention et optimisation de
// l'inference", section "Etape 2: softmax en carreaux"): for every sequence s
// and query head h, out = softmax(q[s,h] . K_s^T * scale) V_s over the
// sequence's context_len tokens, whose K/V rows are gathered through the block
// table (16-token pages).  Query head h reads KV head h / G (G = group size,
// the GQA sharing of "第 10 讲：推理（Inference）").
//
// Design (GB300):
//  * one CTA per (sequence x KV head, partition) -- grid (S*Hkv, parts); the partition is a run of
//    `partition_blocks` 16-token blocks.  All G query heads of the group live
//    in the CTA, so every K/V byte is read from HBM once.
//  * each warp owns a ring of STAGES shared-memory stages and streams its own
//    blocks (round-robin over the partition) with TMA: one 4-D tensor-map load
//    per 64-column half of a block's K (and V), 128-byte swizzled, completing
//    on a per-stage mbarrier.  The block ids of the partition are staged in
//    shared memory once, so no id load sits on the issue path.
//  * QK^T and PV run on the tensor cores as warp-level m16n8k16 bf16 MMAs with
//    fp32 accumulators, transposed so that no MMA row is padding: S^T = K Q^T
//    has a page's 16 keys as M and the G heads as N (8 per n-tile), O^T =
//    V^T P^T has 16 dims per m-tile as M and the heads as N.  At G = 8 this
//    contraction is 8 flop per KV byte, which would keep the fp32 pipe ~70%
//    busy at HBM speed; on the tensor pipe it costs a few percent of its rate.
//    In partitions longer than 256 blocks a warp takes its pages two at a
//    time (two independent chains); in shorter ones one at a time, each ring
//    stage refilled as soon as its page is done.
//  * online softmax in the log2 domain (scores pre-multiplied by
//    scale * log2 e, MUFU ex2); a head's max and sum reduce over the 8 lanes
//    of its column.  P^T enters the PV MMA as bf16 hi + bf16 lo (two MMAs,
//    each 8 x 8 block moved into the B layout by movmatrix.trans), which keeps
//    P's rounding error at ~2^-16 relative instead of bf16's 2^-9.
//  * warps merge in shared memory; a single-partition sequence writes the
//    final output, otherwise the CTA writes its normalised partial output and
//    its log2-sum-exp, and a small merge kernel combines the partitions.
//  * every mbarrier wait is bounded; a timeout sets an error bit, drains the
//    warp's outstanding copies (also bounded) and lets the CTA finish.
#include <algorithm>
#include <climits>
#include <utility>

#include "pkv_decode_body.cuh"
#include "pkv_internal.h"

namespace pkv {

int decode_warps_per_cta() { return kDecodeWarps; }

template <int D, int G, bool PAIR>
__global__ void __launch_bounds__(kDecodeWarps * 32)
paged_decode_split_kernel(const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_v, const DecodeParams p) {
  // inputs may have been written by the previous kernel in the stream (with
  // wait_late: the step's append, waited for only before the last pages)
  if (!p.wait_late) griddep_wait();
  if (p.early_trigger) griddep_launch_dependents();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int pair = blockIdx.x;
  const int part = blockIdx.y;
  const int seq = pair / p.kv_heads;
  const int kvh = pair - seq * p.kv_heads;

  const SeqSpan sp = seq_span(__ldg(p.context_lens + seq), p, seq);
  if (sp.bad && part == 0 && threadIdx.x == 0) atomicOr(&g_decode_error, kErrBadContext);
  const int nparts_s = span_parts(sp, p);
  if (part >= nparts_s) return;
  const size_t row0 = size_t(seq) * p.q_heads + size_t(kvh) * G;  // first output row
  if (sp.count == 0) {  // empty context: zeros
    for (int i = threadIdx.x; i < G * D; i += blockDim.x) store_out(p, row0 * D + i, 0.f);
    return;
  }
  const int b0 = sp.first + part * p.partition_blocks;  // first block of this partition
  const int nb_local = min(sp.first + sp.count - b0, p.partition_blocks);
  const bool final_out = (nparts_s == 1) && !p.force_partials;
  decode_run<D, G, kDecodeWarps, PAIR>(tmap_k, tmap_v, p, smem, seq, kvh, b0, nb_local, sp.len,
                                       final_out, row0 * p.num_parts + part, p.num_parts);
}

// Length-balanced list decode: every CTA computes the same plan from the
// context lengths (list_plan), then takes run blockIdx.x and every
// gridDim.x-th after it.  Block 0 stores the plan for the merge.
template <int D, int G>
__global__ void __launch_bounds__(kDecodeWarps * 32)
paged_decode_list_kernel(const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v, const DecodeParams p,
                         const DecodeListParams lp) {
  griddep_wait();  // inputs may have been written by the previous kernel in the stream
  constexpr int kThreads = kDecodeWarps * 32;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  int32_t* base = reinterpret_cast<int32_t*>(smem + DecodeListTile<D>::kPlanOffset);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int S = lp.num_seqs;
  list_plan<kThreads>(p, lp, base);
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i <= S; i += kThreads) lp.seq_item_base[i] = base[i];
  for (int item = blockIdx.x; item < base[S]; item += gridDim.x) {
    if (item != int(blockIdx.x)) {
      // the previous run is complete: its copies landed and every thread has
      // left its merge; its barriers are retired before they are set up again
      if (lane == 0)
        for (int st = 0; st < kDecodeStages; ++st)
          mbar_inval(smem_u32(smem + DecodeTile<D, kDecodeWarps>::kBarOffset) +
                     (warp * kDecodeStages + st) * 8);
      __syncthreads();
    }
    // one page at a time: the list's CTAs run at the bytes they keep in flight
    // (capped decode of the 70B-GQA batch, GB/s at 32 / 64 / 96 / 152 / 304
    // CTAs: 1493 / 2788 / 4161 / 5845 / 6020 against 1230 / 2271 / 3341 / 4670
    // / 5858 with the pages in pairs)
    list_item<D, G, kDecodeWarps, false>(tmap_k, tmap_v, p, lp, smem, base, item);
  }
}

// The merge of the list's runs: for the row (sequence s, head h), runs
// r < k_s of pair (s, h / G) hold their normalised output and log2-sum-exp
// at partial row (seq_item_base[s] + (h / G) k_s + r) G + h % G; the same
// log-sum-exp merge as paged_decode_merge4_kernel, four dims per thread.
template <int D>
__global__ void __launch_bounds__(256) paged_decode_merge_list_kernel(const DecodeParams p,
                                                                      const DecodeListParams lp,
                                                                      long long total_rows) {
  constexpr int TPR = D / 4;  // threads per row
  griddep_wait();
  const long long gtid = (long long)blockIdx.x * 256 + threadIdx.x;
  const long long row = gtid / TPR;
  const int c4 = int(gtid - row * TPR);
  if (row >= total_rows) return;
  const int seq = int(row / p.q_heads);
  const int h = int(row - (long long)seq * p.q_heads);
  const int G = p.q_heads / p.kv_heads;
  const int kvh = h / G;
  const int b = __ldg(lp.seq_item_base + seq);
  const int runs = (__ldg(lp.seq_item_base + seq + 1) - b) / p.kv_heads;
  const bool extra = has_extra(p, seq);
  if (runs <= 1 && !extra) return;  // written by the decode kernel
  const size_t r0 = size_t(b + kvh * runs) * G + (h - kvh * G);
  float big = extra ? __ldg(p.extra_lse + row) : -INFINITY;
  for (int r = 0; r < runs; ++r) big = fmaxf(big, __ldg(p.part_lse + r0 + size_t(r) * G));
  float tot = 0.f;
  float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
  if (extra) {
    const float w = ex2(__ldg(p.extra_lse + row) - big);
    const float4 x = __ldg(reinterpret_cast<const float4*>(p.extra_o + row * D) + c4);
    tot += w;
    val = make_float4(w * x.x, w * x.y, w * x.z, w * x.w);
  }
#pragma unroll 4
  for (int r = 0; r < runs; ++r) {
    const size_t pr = r0 + size_t(r) * G;
    const float w = ex2(__ldg(p.part_lse + pr) - big);
    const float4 x = __ldg(reinterpret_cast<const float4*>(p.part_o + pr * D) + c4);
    tot += w;
    val.x += w * x.x;
    val.y += w * x.y;
    val.z += w * x.z;
    val.w += w * x.w;
  }
  const float4 res = tot > 0.f ? make_float4(val.x / tot, val.y / tot, val.z / tot, val.w / tot)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
  const size_t o = size_t(row) * D + size_t(c4) * 4;
  store_out(p, o, res.x);
  store_out(p, o + 1, res.y);
  store_out(p, o + 2, res.z);
  store_out(p, o + 3, res.w);
}

// Log-sum-exp merge of the partitions of one (sequence, query head): with
// lse_p the log2-sum-exp of partition p and o_p its normalised output,
// out = sum_p 2^(lse_p - M) o_p / sum_p 2^(lse_p - M), M = max_p lse_p.
template <int D>
__global__ void __launch_bounds__(D) paged_decode_merge_kernel(const DecodeParams p) {
  griddep_wait();
  const size_t row = blockIdx.x;  // seq * q_heads + head
  const int seq = int(row / p.q_heads);
  const SeqSpan sp = seq_span(__ldg(p.context_lens + seq), p, seq);
  const int nparts_s = span_parts(sp, p);
  const bool extra = has_extra(p, seq);
  if (nparts_s == 1 && !p.force_partials) return;  // written by the split kernel
  const float* lse = p.part_lse + row * p.num_parts;
  const float* po = p.part_o + row * p.num_parts * D + threadIdx.x;
  float big = extra ? __ldg(p.extra_lse + row) : -INFINITY;
  for (int q = 0; q < nparts_s; ++q) big = fmaxf(big, __ldg(lse + q));
  float tot = 0.f, val = 0.f;
  if (extra) {
    const float w = ex2(__ldg(p.extra_lse + row) - big);
    tot += w;
    val += w * __ldg(p.extra_o + row * D + threadIdx.x);
  }
#pragma unroll 4
  for (int q = 0; q < nparts_s; ++q) {
    const float w = ex2(__ldg(lse + q) - big);
    tot += w;
    val += w * __ldg(po + size_t(q) * D);
  }
  store_out(p, row * D + threadIdx.x, tot > 0.f ? val / tot : 0.f);
}

// The same merge with one warp-sized group of threads per row, each thread
// four consecutive dims as float4 (out 16-byte aligned): a quarter of the
// CTAs of the scalar form and four partial values in flight per load.
template <int D>
__global__ void __launch_bounds__(256) paged_decode_merge4_kernel(const DecodeParams p,
                                                                  long long total_rows) {
  constexpr int TPR = D / 4;  // threads per row
  griddep_wait();
  const long long gtid = (long long)blockIdx.x * 256 + threadIdx.x;
  const long long row = gtid / TPR;
  const int c4 = int(gtid - row * TPR);
  if (row >= total_rows) return;
  const int seq = int(row / p.q_heads);
  const SeqSpan sp = seq_span(__ldg(p.context_lens + seq), p, seq);
  const int nparts_s = span_parts(sp, p);
  const bool extra = has_extra(p, seq);
  if (nparts_s == 1 && !p.force_partials) return;  // written by the split kernel
  const float* lse = p.part_lse + row * p.num_parts;
  const float4* po = reinterpret_cast<const float4*>(p.part_o + row * p.num_parts * D) + c4;
  float big = extra ? __ldg(p.extra_lse + row) : -INFINITY;
  for (int q = 0; q < nparts_s; ++q) big = fmaxf(big, __ldg(lse + q));
  float tot = 0.f;
  float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
  if (extra) {
    const float w = ex2(__ldg(p.extra_lse + row) - big);
    const float4 x = __ldg(reinterpret_cast<const float4*>(p.extra_o + row * D) + c4);
    tot += w;
    val = make_float4(w * x.x, w * x.y, w * x.z, w * x.w);
  }
#pragma unroll 4
  for (int q = 0; q < nparts_s; ++q) {
    const float w = ex2(__ldg(lse + q) - big);
    const float4 x = __ldg(po + size_t(q) * TPR);
    tot += w;
    val.x += w * x.x;
    val.y += w * x.y;
    val.z += w * x.z;
    val.w += w * x.w;
  }
  // the same division as the scalar form, so both give the same bits
  const float4 res = tot > 0.f ? make_float4(val.x / tot, val.y / tot, val.z / tot, val.w / tot)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
  if (p.out_bf16) {  // four bf16 (8 bytes; out 8-byte aligned)
    __nv_bfloat162 lo = __floats2bfloat162_rn(res.x, res.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(res.z, res.w);
    uint2 v;
    v.x = *reinterpret_cast<uint32_t*>(&lo);
    v.y = *reinterpret_cast<uint32_t*>(&hi);
    reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.out) + row * D)[c4] = v;
  } else {
    reinterpret_cast<float4*>(p.out + row * D)[c4] = res;
  }
}

// Partitions longer than this take their pages in pairs (two MMA and
// exponential chains per warp), shorter ones one at a time (each stage
// refilled as soon as its page is done).  Same box, 70B-GQA recipe, decode
// step, pairs / single: 8 sequences (90-block partitions) 39.7 / 38.5 us,
// 12 (about 160) 48.0 / 44.6 us, 256 (384) within 0.4%; 128K contexts
// (1024-block partitions) 318.5 / 328.6 us.
constexpr int kSplitPairMinBlocks = 256;

template <int D, int G, bool PAIR>
static cudaError_t launch_split_t(const DecodeParams& prm, int num_seqs,
                                  const CUtensorMap* tmap_k, const CUtensorMap* tmap_v,
                                  cudaStream_t stream) {
  using T = DecodeTile<D, kDecodeWarps>;
  static std::atomic<int> attr_done[kAttrMaxDevices];
  {
    const cudaError_t e =
        set_smem_limit_once(paged_decode_split_kernel<D, G, PAIR>, T::kSmemBytes, attr_done);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(num_seqs * prm.kv_heads, prm.num_parts);
  return launch_after_previous(paged_decode_split_kernel<D, G, PAIR>, grid,
                               dim3(kDecodeWarps * 32), T::kSmemBytes, stream, *tmap_k, *tmap_v,
                               prm);
}

template <int D, int G>
static cudaError_t launch_decode_t(const DecodeParams& prm, int num_seqs,
                                   const CUtensorMap* tmap_k, const CUtensorMap* tmap_v,
                                   cudaStream_t stream, bool with_merge) {
  const cudaError_t e =
      prm.partition_blocks > kSplitPairMinBlocks
          ? launch_split_t<D, G, true>(prm, num_seqs, tmap_k, tmap_v, stream)
          : launch_split_t<D, G, false>(prm, num_seqs, tmap_k, tmap_v, stream);
  if (e != cudaSuccess || !with_merge) return e;
  return launch_decode_merge(prm, num_seqs, D, stream);
}

template <int D, int G>
static cudaError_t launch_decode_list_t(const DecodeParams& prm, const DecodeListParams& lp,
                                        int items, int max_ctas, const CUtensorMap* tmap_k,
                                        const CUtensorMap* tmap_v, cudaStream_t stream) {
  using L = DecodeListTile<D>;
  static std::atomic<int> attr_done[kAttrMaxDevices];
  cudaError_t e = set_smem_limit_once(paged_decode_list_kernel<D, G>, L::kSmemBytes, attr_done);
  if (e != cudaSuccess) return e;
  const int ctas = max_ctas > 0 && max_ctas < items ? max_ctas : items;
  e = launch_after_previous(paged_decode_list_kernel<D, G>, dim3(unsigned(ctas)),
                            dim3(kDecodeWarps * 32), L::kSmemBytes, stream, *tmap_k, *tmap_v, prm,
                            lp);
  if (e != cudaSuccess) return e;
  return launch_decode_list_merge(prm, lp, D, stream);
}

cudaError_t launch_decode_list_merge(const DecodeParams& prm, const DecodeListParams& lp,
                                     int d_head, cudaStream_t stream) {
  const long long rows = (long long)lp.num_seqs * prm.q_heads;
  const long long blocks = (rows * (d_head / 4) + 255) / 256;
  if (blocks > INT32_MAX) return cudaErrorInvalidValue;
  if (d_head == 128)
    return launch_after_previous(paged_decode_merge_list_kernel<128>, dim3(unsigned(blocks)),
                                 dim3(256), 0, stream, prm, lp, rows);
  if (d_head == 64)
    return launch_after_previous(paged_decode_merge_list_kernel<64>, dim3(unsigned(blocks)),
                                 dim3(256), 0, stream, prm, lp, rows);
  return cudaErrorInvalidValue;
}

template <int D>
static cudaError_t launch_decode_list_d(const DecodeParams& prm, const DecodeListParams& lp,
                                        int items, int max_ctas, int group, const CUtensorMap* tk,
                                        const CUtensorMap* tv, cudaStream_t st) {
  switch (group) {
    case 1: return launch_decode_list_t<D, 1>(prm, lp, items, max_ctas, tk, tv, st);
    case 2: return launch_decode_list_t<D, 2>(prm, lp, items, max_ctas, tk, tv, st);
    case 4: return launch_decode_list_t<D, 4>(prm, lp, items, max_ctas, tk, tv, st);
    case 8: return launch_decode_list_t<D, 8>(prm, lp, items, max_ctas, tk, tv, st);
    case 16: return launch_decode_list_t<D, 16>(prm, lp, items, max_ctas, tk, tv, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_merge(const DecodeParams& prm, int num_seqs, int d_head,
                                cudaStream_t stream) {
  if (prm.num_parts == 1 && !prm.force_partials) return cudaSuccess;
  const long long rows = (long long)num_seqs * prm.q_heads;
  const uintptr_t vec_align = prm.out_bf16 ? 7 : 15;  // four outputs per thread
  const bool vec = (reinterpret_cast<uintptr_t>(prm.out) & vec_align) == 0;
  if (vec && (d_head == 128 || d_head == 64)) {
    const long long blocks = (rows * (d_head / 4) + 255) / 256;
    if (blocks > INT32_MAX) return cudaErrorInvalidValue;
    if (d_head == 128)
      return launch_after_previous(paged_decode_merge4_kernel<128>, dim3(unsigned(blocks)),
                                   dim3(256), 0, stream, prm, rows);
    return launch_after_previous(paged_decode_merge4_kernel<64>, dim3(unsigned(blocks)), dim3(256),
                                 0, stream, prm, rows);
  } else if (d_head == 128) {
    return launch_after_previous(paged_decode_merge_kernel<128>,
                                 dim3(unsigned(num_seqs * prm.q_heads)), dim3(128), 0, stream, prm);
  } else if (d_head == 64) {
    return launch_after_previous(paged_decode_merge_kernel<64>,
                                 dim3(unsigned(num_seqs * prm.q_heads)), dim3(64), 0, stream, prm);
  }
  return cudaErrorInvalidValue;
}

template <int D>
static cudaError_t launch_decode_d(const DecodeParams& prm, int num_seqs, int group,
                                   const CUtensorMap* tk, const CUtensorMap* tv,
                                   cudaStream_t st, bool with_merge) {
  switch (group) {
    case 1: return launch_decode_t<D, 1>(prm, num_seqs, tk, tv, st, with_merge);
    case 2: return launch_decode_t<D, 2>(prm, num_seqs, tk, tv, st, with_merge);
    case 4: return launch_decode_t<D, 4>(prm, num_seqs, tk, tv, st, with_merge);
    case 8: return launch_decode_t<D, 8>(prm, num_seqs, tk, tv, st, with_merge);
    case 16: return launch_decode_t<D, 16>(prm, num_seqs, tk, tv, st, with_merge);
    default: return cudaErrorInvalidValue;
  }
}

static DecodeParams decode_params(const DecodeArgs& a) {
  DecodeParams prm;
  prm.q = static_cast<const __nv_bfloat16*>(a.q);
  prm.block_tables = a.block_tables;
  prm.context_lens = a.context_lens;
  prm.out = a.out;
  prm.part_o = a.part_o;
  prm.part_lse = a.part_lse;
  prm.q_heads = a.q_heads;
  prm.kv_heads = a.kv_heads;
  prm.num_blocks = a.num_blocks;
  prm.max_blocks_per_seq = a.max_blocks_per_seq;
  prm.partition_blocks = a.partition_blocks;
  prm.num_parts = a.num_parts;
  prm.scale_log2 = a.scale_log2;
  prm.out_scale = 1.f;
  prm.first_block = a.first_block;
  prm.force_partials = a.force_partials;
  prm.extra_o = a.extra_o;
  prm.extra_lse = a.extra_lse;
  prm.out_bf16 = a.out_bf16 ? 1 : 0;
  prm.seq_first_block = a.seq_first_block;
  prm.early_trigger = a.early_trigger ? 1 : 0;
  prm.wait_late = a.wait_late ? 1 : 0;
  prm.step_slots = a.step_slots;
  return prm;
}

cudaError_t launch_paged_decode_merge_only(const DecodeArgs& a, cudaStream_t stream) {
  return launch_decode_merge(decode_params(a), a.num_seqs, a.d_head, stream);
}

cudaError_t launch_paged_decode(const DecodeArgs& a, const CUtensorMap* tmap_k,
                                const CUtensorMap* tmap_v, cudaStream_t stream) {
  const DecodeParams prm = decode_params(a);
  const bool with_merge = !a.skip_merge;
  const int group = a.q_heads / a.kv_heads;
  if (a.list) {
    if (a.num_seqs > kListMaxSeqs || a.list_items <= 0) return cudaErrorInvalidValue;
    DecodeListParams lp;
    lp.seq_item_base = a.list_base;
    lp.num_seqs = a.num_seqs;
    lp.target_items = a.list_target;
    lp.min_run = a.list_min_run;
    lp.max_blocks = a.list_max_blocks;
    if (a.d_head == 128)
      return launch_decode_list_d<128>(prm, lp, a.list_items, a.list_max_ctas, group, tmap_k,
                                       tmap_v, stream);
    if (a.d_head == 64)
      return launch_decode_list_d<64>(prm, lp, a.list_items, a.list_max_ctas, group, tmap_k,
                                      tmap_v, stream);
    return cudaErrorInvalidValue;
  }
  if (a.d_head == 128)
    return launch_decode_d<128>(prm, a.num_seqs, group, tmap_k, tmap_v, stream, with_merge);
  if (a.d_head == 64)
    return launch_decode_d<64>(prm, a.num_seqs, group, tmap_k, tmap_v, stream, with_merge);
  return cudaErrorInvalidValue;
}

// Prefix groups (see launch_prefix_groups_setup): one warp per sequence (its
// lanes compare the prefix ids 32 at a time), then one thread per group.
__global__ void prefix_groups_setup_kernel(const int32_t* group_start,
                                           const int32_t* group_prefix_blocks, int num_groups,
                                           int uniform_prefix_blocks, int num_seqs,
                                           const int32_t* block_tables, int max_blocks,
                                           const int32_t* context_lens, int max_prefix_blocks,
                                           int32_t* seq_first_block, int32_t* group_ctx) {
  griddep_wait();
  const bool uniform = group_start == nullptr;
  const int groups = uniform ? 1 : num_groups;
  const int lane = threadIdx.x & 31;
  auto prefix_of = [&](int g) {
    const int pb = uniform ? uniform_prefix_blocks : __ldg(group_prefix_blocks + g);
    return (pb >= 1 && pb <= max_prefix_blocks && pb <= max_blocks) ? pb : 0;
  };
  const long long threads = (long long)gridDim.x * blockDim.x;
  const long long gtid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  // a group's prefix length in tokens
  for (long long g = gtid; g < groups; g += threads) group_ctx[g] = prefix_of(int(g)) * kBlockTokens;
  const long long warps = threads / 32;
  for (long long w = gtid / 32; w < num_seqs; w += warps) {
    const int s = int(w);
    int g = 0, lead = 0;
    bool in_group = true;
    if (!uniform) {  // the last group starting at or before s
      int lo = 0, hi = num_groups - 1;
      in_group = num_groups > 0 && __ldg(group_start) <= s;
      while (in_group && lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(group_start + mid) <= s) lo = mid;
        else hi = mid - 1;
      }
      g = lo;
      lead = in_group ? __ldg(group_start + g) : 0;
      in_group = in_group && s < __ldg(group_start + g + 1) && lead >= 0;
    }
    int pb = in_group ? prefix_of(g) : 0;
    bool bad = in_group && pb == 0;  // a group whose prefix length is out of range
    if (pb > 0 && __ldg(context_lens + s) < pb * kBlockTokens) {
      pb = 0;  // the prefix is longer than the context
      bad = true;
    }
    if (pb > 0 && s != lead) {
      const int32_t* mine = block_tables + size_t(s) * max_blocks;
      const int32_t* theirs = block_tables + size_t(lead) * max_blocks;
      bool same = true;
      for (int j = lane; j < pb; j += 32) same = same && __ldg(mine + j) == __ldg(theirs + j);
      if (!__all_sync(0xffffffffu, same)) {
        pb = 0;
        bad = true;
      }
    }
    if (lane == 0) {
      if (bad) atomicOr(&g_decode_error, kErrPrefixMismatch);
      seq_first_block[s] = pb;
    }
  }
}

cudaError_t launch_prefix_groups_setup(const int32_t* group_start,
                                       const int32_t* group_prefix_blocks, int num_groups,
                                       int uniform_prefix_blocks, int num_seqs,
                                       const int32_t* block_tables, int max_blocks_per_seq,
                                       const int32_t* context_lens, int max_prefix_blocks,
                                       int32_t* seq_first_block, int32_t* group_ctx,
                                       cudaStream_t stream) {
  const long long warps = (long long)num_seqs > (group_start ? num_groups : 1)
                              ? num_seqs : (group_start ? num_groups : 1);
  const int blocks = int(std::min<long long>((warps * 32 + 255) / 256, 1024));
  return launch_after_previous(prefix_groups_setup_kernel, dim3(blocks), dim3(256), 0, stream,
                               group_start, group_prefix_blocks, num_groups,
                               uniform_prefix_blocks, num_seqs, block_tables, max_blocks_per_seq,
                               context_lens, max_prefix_blocks, seq_first_block, group_ctx);
}

int decode_max_partition_blocks() { return kMaxPartitionBlocks; }
int decode_list_max_seqs() { return kListMaxSeqs; }

// Device address of this unit's error word on the current device.
cudaError_t decode_error_word(unsigned** word) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(word), g_decode_error);
}

unsigned read_decode_error(bool clear) {
  unsigned word = 0;
  if (cudaMemcpyFromSymbol(&word, g_decode_error, sizeof(word)) != cudaSuccess) return ~0u;
  if (clear) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_decode_error, &zero, sizeof(zero)) != cudaSuccess) return ~0u;
  }
  return word;
}

}  // namespace pkv
