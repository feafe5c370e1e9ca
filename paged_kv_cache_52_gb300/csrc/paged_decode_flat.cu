// Flat split of the paged decode (bf16 or FP8 pools).  The blocks of all
// sequences are laid end to end and cut into equal ranges, one per group of Hkv warps of a
// persistent grid (one CTA per SM); warp h of a group streams KV head h of
// its group's range.  The ranges differ by at most one block, so every warp
// finishes at about the same time whatever the lengths; a warp's ring of page
// copies runs on across the sequence boundaries inside its range, so the
// pipeline fills once per warp instead of once per partition; and the warps
// of a group read the heads of the same blocks side by side, as the uniform
// split's CTAs of one partition do.  A warp holding a whole (sequence, head)
// pair writes its output; the pieces of a pair split between groups are
// written as normalised partials with their log2-sum-exp and combined by the
// flat merge (the same log-sum-exp merge as the uniform split's).  The
// per-page arithmetic is the decode bodies' (bf16_pages, fp8_pages).  In the
// shared-prefix (cascade) decode a sequence's own blocks start after its
// prefix (first_block_of), every piece of a sequence with a prefix part is
// written as a partial, and the merge folds the prefix part in.

#include <atomic>
#include <climits>
#include <type_traits>

#include "pkv_decode_flat_body.cuh"
#include "pkv_internal.h"

namespace pkv {

constexpr int kFlatMaxSeqs = 1024;

// A flat CTA by page format: bf16 pages (the decode body's 3-stage rings of
// one 2 x 16 x D x 2-byte page per stage) or FP8 pages (4 stages of 4 KB of
// e4m3 codes, d_head 128); as many ring-owning warps as one SM's shared
// memory holds beside the plan.
template <int D, bool FP8>
struct FlatCfg {
  static constexpr int NW = FP8 ? 12 : (D == 128 ? 9 : 16);
  static constexpr int kStages = FlatPage<D, FP8>::kStages;
  static constexpr int kRingBytes = FlatPage<D, FP8>::kRingBytes;
  static constexpr int kBarOffset = NW * kRingBytes;
  static constexpr int kPreOffset = kBarOffset + NW * kStages * 8;  // [kFlatMaxSeqs + 1] prefix sums
  static constexpr int kScanOffset = kPreOffset + (kFlatMaxSeqs + 1) * 4;  // per-warp totals
  static constexpr int kEnd = kScanOffset + 32 * 4;
  static constexpr int kSmemBytes = kEnd + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 232448, "flat decode CTA does not fit in shared memory");
  static_assert(!FP8 || D == kF8D, "the FP8 pages are d_head 128");
};

template <int D, int G, bool FP8>
__global__ void __launch_bounds__(FlatCfg<D, FP8>::NW * 32, 1)
paged_decode_flat_kernel(const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v, const DecodeParams p,
                         const DecodeFlatParams fp) {
  using F = FlatCfg<D, FP8>;
  using T = F;
  constexpr int NW = F::NW;
  constexpr int kStages = F::kStages;
  constexpr int kThreads = NW * 32;
  constexpr unsigned kFull = 0xffffffffu;
  // with wait_late only the loads of a sequence's last page wait for the
  // grid before (the step's append); otherwise every input may be its output
  if (!p.wait_late) griddep_wait();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  int32_t* pre = reinterpret_cast<int32_t*>(smem + F::kPreOffset);
  int32_t* scan = reinterpret_cast<int32_t*>(smem + F::kScanOffset);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int S = fp.num_seqs;
  const int Hkv = p.kv_heads;

  // ---- the plan, computed alike by every CTA: pages per sequence and their
  // exclusive prefix sum pre[], pre[S] the pages of one KV head
  const int per = (S + kThreads - 1) / kThreads;
  const int s_begin = threadIdx.x * per;
  int local = 0;
  for (int k = 0; k < per; ++k) {
    const int s = s_begin + k;
    if (s < S) {
      bool bad;
      int first;
      const int n = flat_own_pages(p, s, fp.max_blocks, first, bad);
      if (bad && blockIdx.x == 0) atomicOr(&g_decode_error, kErrBadContext);
      pre[s] = n;
      local += n;
    }
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) scan[warp] = incl;
  const uint32_t ring = smem_u32(smem + warp * T::kRingBytes);
  const uint32_t bars = smem_u32(smem + T::kBarOffset) + warp * kStages * 8;
  if (lane == 0) {
    for (int st = 0; st < kStages; ++st) mbar_init(bars + st * 8, 1);
    fence_barrier_init();
  }
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_v);
  }
  __syncthreads();
  if (warp == 0) {
    int v = lane < NW ? scan[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(kFull, v, o);
      if (lane >= o) v += u;
    }
    if (lane < NW) scan[lane] = v;  // inclusive over the warps
  }
  __syncthreads();
  {
    int base = (warp > 0 ? scan[warp - 1] : 0) + incl - local;
    for (int k = 0; k < per; ++k) {
      const int s = s_begin + k;
      if (s < S) {
        const int n = pre[s];
        pre[s] = base;
        base += n;
      }
    }
    if (threadIdx.x == 0) pre[S] = scan[NW - 1];
  }
  __syncthreads();
  if (blockIdx.x == 0)
    for (int s = threadIdx.x; s <= S; s += kThreads) fp.pre_out[s] = pre[s];

  // ---- this warp's range [f0, f1) of the blocks laid end to end (sequence
  // s holds offsets pre[s] + b, b < n_s): its group's, in KV head hw
  const long long total = pre[S];
  const long long groups = flat_groups((long long)gridDim.x * NW, Hkv);
  const long long gw = (long long)blockIdx.x * NW + warp;
  const long long g = gw / Hkv;
  const int hw = int(gw - g * Hkv);
  const long long c = flat_chunk(total, groups, fp.min_pages);
  const long long f0 = g * c;
  const long long f1 = g >= groups ? f0 : (f0 + c < total ? f0 + c : total);
  // (a warp with no range returns at once: no CTA-wide barrier follows)

  flat_range<D, G, FP8>(tmap_k, tmap_v, p, pre, S, f0, f1, g, hw, ring, bars);
}

// The merge of the flat split: row (sequence s, head hq) of KV head h =
// hq / G; the sequence's own blocks [pre[s], pre[s] + n_s) in the order of
// the launch lie in the ranges of groups w0 = pre[s] / c .. w1 = (pre[s] +
// n_s - 1) / c, and group w's piece is at partial slot (s + w) Hkv + h.  A
// pair inside one group's range, without a prefix part, was written by the
// kernel; in the cascade decode the prefix part (extra_o, extra_lse) is one
// more piece; an empty sequence without one gets zeros.  The D / 4 threads of
// a row (a warp at d_head 128, half a warp at 64) each own four dims; a
// small batch splits a pair into many pieces, so the threads first take the
// pieces' log2-sum-exps in turn (max and weight sum reduced over the row's
// threads), then each accumulates its dims over every piece with eight loads
// in flight.
template <int D>
__global__ void __launch_bounds__(256) paged_decode_merge_flat_kernel(const DecodeParams p,
                                                                      const DecodeFlatParams fp,
                                                                      long long total_rows) {
  constexpr int TPR = D / 4;  // threads per row: 32 or 16, a warp's aligned lanes
  griddep_wait();
  const long long gtid = (long long)blockIdx.x * 256 + threadIdx.x;
  const long long row = gtid / TPR;
  const int c4 = int(gtid - row * TPR);
  // no early return before the shuffles: a warp's rows run them together
  const bool valid = row < total_rows;
  long long w0 = 0, w1 = -1;
  int hg = 0, h = 0, seq = 0;
  bool extra = false;
  if (valid) {
    seq = int(row / p.q_heads);
    const int hq = int(row - (long long)seq * p.q_heads);
    const int G = p.q_heads / p.kv_heads;
    h = hq / G;
    hg = hq - h * G;
    extra = has_extra(p, seq);
    const int32_t* pre = fp.pre_out;
    const int n = __ldg(pre + seq + 1) - __ldg(pre + seq);
    if (n > 0) {
      const long long total = __ldg(pre + fp.num_seqs);
      const long long c =
          fp.chunk > 0 ? fp.chunk
                       : flat_chunk(total, flat_groups(fp.total_warps, p.kv_heads), fp.min_pages);
      const long long start = __ldg(pre + seq);
      w0 = start / c;
      w1 = (start + n - 1) / c;
    }
  }
  const bool pieces = w1 >= w0;
  const bool merge = extra || w1 > w0;  // else written by the kernel, or zeros
  const int G = p.q_heads / p.kv_heads;
  auto slot_of = [&](long long w) { return (size_t(seq + w) * p.kv_heads + h) * G + hg; };
  auto lse_of = [&](long long w) { return __ldg(p.part_lse + slot_of(w)); };
  float big = -INFINITY;
  if (merge && pieces)
    for (long long w = w0 + c4; w <= w1; w += TPR) big = fmaxf(big, lse_of(w));
#pragma unroll
  for (int o = TPR / 2; o > 0; o >>= 1) big = fmaxf(big, __shfl_xor_sync(0xffffffffu, big, o));
  const float xl = (valid && extra) ? __ldg(p.extra_lse + row) : -INFINITY;
  big = fmaxf(big, xl);
  float tot = 0.f;
  if (merge && pieces)
    for (long long w = w0 + c4; w <= w1; w += TPR) tot += ex2(lse_of(w) - big);
#pragma unroll
  for (int o = TPR / 2; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  if (!valid || (!merge && pieces)) return;  // outside the batch, or written by the kernel
  float4 res = make_float4(0.f, 0.f, 0.f, 0.f);
  if (merge) {
    float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
    if (extra) {
      const float wgt = ex2(xl - big);
      const float4 x = __ldg(reinterpret_cast<const float4*>(p.extra_o + size_t(row) * D) + c4);
      tot += wgt;
      val = make_float4(wgt * x.x, wgt * x.y, wgt * x.z, wgt * x.w);
    }
#pragma unroll 8
    for (long long w = w0; w <= w1; ++w) {
      const size_t slot = slot_of(w);
      const float wgt = ex2(__ldg(p.part_lse + slot) - big);
      const float4 x = __ldg(reinterpret_cast<const float4*>(p.part_o + slot * D) + c4);
      val.x += wgt * x.x;
      val.y += wgt * x.y;
      val.z += wgt * x.z;
      val.w += wgt * x.w;
    }
    res = make_float4(val.x / tot, val.y / tot, val.z / tot, val.w / tot);
  }
  const size_t o = size_t(row) * D + 4 * c4;
  store_out(p, o, res.x);
  store_out(p, o + 1, res.y);
  store_out(p, o + 2, res.z);
  store_out(p, o + 3, res.w);
}

template <int D>
static cudaError_t launch_flat_merge_t(const DecodeParams& prm, const DecodeFlatParams& fp,
                                       cudaStream_t stream) {
  const long long rows = (long long)fp.num_seqs * prm.q_heads;
  const long long blocks = (rows * (D / 4) + 255) / 256;
  if (blocks > INT32_MAX) return cudaErrorInvalidValue;
  return launch_after_previous(paged_decode_merge_flat_kernel<D>, dim3(unsigned(blocks)),
                               dim3(256), 0, stream, prm, fp, rows);
}

template <int D, int G, bool FP8>
static cudaError_t launch_flat_t(const DecodeParams& prm, const DecodeFlatParams& fp, int ctas,
                                 const CUtensorMap* tk, const CUtensorMap* tv,
                                 cudaStream_t stream, bool with_merge) {
  using F = FlatCfg<D, FP8>;
  static std::atomic<int> attr_done[kAttrMaxDevices];
  cudaError_t e =
      set_smem_limit_once(paged_decode_flat_kernel<D, G, FP8>, F::kSmemBytes, attr_done);
  if (e != cudaSuccess) return e;
  e = launch_after_previous(paged_decode_flat_kernel<D, G, FP8>, dim3(unsigned(ctas)),
                            dim3(F::NW * 32), F::kSmemBytes, stream, *tk, *tv, prm, fp);
  if (e != cudaSuccess || !with_merge) return e;
  return launch_flat_merge_t<D>(prm, fp, stream);
}

template <int D, bool FP8>
static cudaError_t launch_flat_d(const DecodeParams& prm, const DecodeFlatParams& fp, int group,
                                 int ctas, const CUtensorMap* tk, const CUtensorMap* tv,
                                 cudaStream_t st, bool with_merge) {
  switch (group) {
    case 1: return launch_flat_t<D, 1, FP8>(prm, fp, ctas, tk, tv, st, with_merge);
    case 2: return launch_flat_t<D, 2, FP8>(prm, fp, ctas, tk, tv, st, with_merge);
    case 4: return launch_flat_t<D, 4, FP8>(prm, fp, ctas, tk, tv, st, with_merge);
    case 8: return launch_flat_t<D, 8, FP8>(prm, fp, ctas, tk, tv, st, with_merge);
    case 16: return launch_flat_t<D, 16, FP8>(prm, fp, ctas, tk, tv, st, with_merge);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_flat_merge(const DecodeParams& prm, const DecodeFlatParams& fp,
                                     int d_head, cudaStream_t stream) {
  if (d_head == 128) return launch_flat_merge_t<128>(prm, fp, stream);
  if (d_head == 64) return launch_flat_merge_t<64>(prm, fp, stream);
  return cudaErrorInvalidValue;
}

int decode_flat_warps(int d_head, bool fp8) {
  if (fp8) return d_head == kF8D ? FlatCfg<kF8D, true>::NW : 0;
  return d_head == 128 ? FlatCfg<128, false>::NW : d_head == 64 ? FlatCfg<64, false>::NW : 0;
}
int decode_flat_max_seqs() { return kFlatMaxSeqs; }

// The kernel's and the merge's parameters from the launch arguments.
static bool flat_params(const DecodeArgs& a, DecodeParams& prm, DecodeFlatParams& fp) {
  if (a.num_seqs <= 0 || a.num_seqs > kFlatMaxSeqs || a.flat_ctas <= 0 || !a.flat_pre ||
      !a.part_o || !a.part_lse || decode_flat_warps(a.d_head, a.fp8) == 0)
    return false;
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
  prm.partition_blocks = 0;  // not used by the flat split
  prm.num_parts = 0;
  prm.scale_log2 = a.scale_log2;
  prm.out_scale = a.fp8 ? a.out_scale : 1.f;
  prm.first_block = a.first_block;
  prm.force_partials = 0;
  prm.extra_o = a.extra_o;
  prm.extra_lse = a.extra_lse;
  prm.out_bf16 = a.out_bf16 ? 1 : 0;
  prm.seq_first_block = a.seq_first_block;
  prm.wait_late = a.wait_late ? 1 : 0;
  prm.step_slots = a.step_slots;
  fp.pre_out = a.flat_pre;
  fp.num_seqs = a.num_seqs;
  fp.max_blocks = a.flat_max_blocks;
  fp.total_warps = a.flat_ctas * decode_flat_warps(a.d_head, a.fp8);
  fp.min_pages = kFlatMinPages;
  return true;
}

cudaError_t launch_paged_decode_flat(const DecodeArgs& a, const CUtensorMap* tmap_k,
                                     const CUtensorMap* tmap_v, cudaStream_t stream) {
  DecodeParams prm;
  DecodeFlatParams fp;
  if (!flat_params(a, prm, fp)) return cudaErrorInvalidValue;
  const int group = a.q_heads / a.kv_heads;
  const bool with_merge = !a.skip_merge;
  if (a.fp8)
    return launch_flat_d<kF8D, true>(prm, fp, group, a.flat_ctas, tmap_k, tmap_v, stream,
                                      with_merge);
  if (a.d_head == 128)
    return launch_flat_d<128, false>(prm, fp, group, a.flat_ctas, tmap_k, tmap_v, stream,
                                     with_merge);
  return launch_flat_d<64, false>(prm, fp, group, a.flat_ctas, tmap_k, tmap_v, stream,
                                  with_merge);
}

cudaError_t launch_paged_decode_flat_merge(const DecodeArgs& a, cudaStream_t stream) {
  DecodeParams prm;
  DecodeFlatParams fp;
  if (!flat_params(a, prm, fp)) return cudaErrorInvalidValue;
  if (a.d_head == 128) return launch_flat_merge_t<128>(prm, fp, stream);
  return launch_flat_merge_t<64>(prm, fp, stream);
}

// Device address of this unit's error word on the current device.
cudaError_t decode_flat_error_word(unsigned** word) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(word), g_decode_error);
}

unsigned read_decode_flat_error(bool clear) {
  unsigned word = 0;
  if (cudaMemcpyFromSymbol(&word, g_decode_error, sizeof(word)) != cudaSuccess) return ~0u;
  if (clear) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_decode_error, &zero, sizeof(zero)) != cudaSuccess) return ~0u;
  }
  return word;
}

}  // namespace pkv
