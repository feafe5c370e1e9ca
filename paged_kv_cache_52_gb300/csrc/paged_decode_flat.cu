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

#include "pkv_decode_body.cuh"
#include "pkv_decode_fp8_body.cuh"
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
  static constexpr int kStages = FP8 ? 4 : kDecodeStages;
  static constexpr int kStageBytes = FP8 ? F8Page::kStageBytes : DecodeTile<D, NW>::kStageBytes;
  static constexpr int kTileBytes = kStageBytes / 2;   // K, then V
  static constexpr int kHalfBytes = kBlockTokens * 128;  // a 64-dim bf16 half of a tile
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kBarOffset = NW * kRingBytes;
  static constexpr int kPreOffset = kBarOffset + NW * kStages * 8;  // [kFlatMaxSeqs + 1] prefix sums
  static constexpr int kScanOffset = kPreOffset + (kFlatMaxSeqs + 1) * 4;  // per-warp totals
  static constexpr int kEnd = kScanOffset + 32 * 4;
  static constexpr int kSmemBytes = kEnd + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 232448, "flat decode CTA does not fit in shared memory");
  static_assert(!FP8 || D == kF8D, "the FP8 pages are d_head 128");
};

// Blocks a group takes at least: a shorter range would not amortise its
// warps' start (the plan, block ids and first copies) and would only add
// pieces to merge.
constexpr int kFlatMinPages = 8;

struct DecodeFlatParams {
  int32_t* pre_out;  // [num_seqs + 1] the block prefix sums, for the merge
  int num_seqs;      // <= kFlatMaxSeqs
  int max_blocks;    // blocks attended per sequence at most
  int total_warps;   // warps of the launch
  int min_pages;     // blocks per group at least (the last busy group may take fewer)
};

// Groups of a launch: its warps in groups of Hkv (the rest idle).
__device__ __forceinline__ long long flat_groups(long long warps, int kv_heads) {
  return warps / kv_heads;
}

// Blocks per group: the blocks of all sequences shared out over the groups,
// at least min_pages each (the merge must use the same value).
__device__ __forceinline__ long long flat_chunk(long long total, long long groups, int min_pages) {
  const long long c = total > 0 ? (total + groups - 1) / groups : 1;
  return c > min_pages ? c : min_pages;
}

// Pages of a context of `len` tokens, clamped to `max_blocks` (bad: the
// length was negative or had to be clamped).
__device__ __forceinline__ int flat_pages(int len, int max_blocks, bool& bad) {
  bad = len < 0;
  int n = len <= 0 ? 0 : len / kBlockTokens + (len % kBlockTokens != 0);
  if (n > max_blocks) {
    n = max_blocks;
    bad = true;
  }
  return n;
}

// A sequence's own pages: those after its first own block (0 without a
// shared prefix), and that block.
__device__ __forceinline__ int flat_own_pages(const DecodeParams& p, int seq, int max_blocks,
                                              int& first, bool& bad) {
  const int len = __ldg(p.context_lens + seq);
  const int n = flat_pages(len, max_blocks, bad);
  first = p.seq_first_block ? __ldg(p.seq_first_block + seq) : p.first_block;
  if (first > 0 && len < first * kBlockTokens) bad = true;  // shorter than its prefix
  return n > first ? n - first : 0;
}

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
  using Acc = std::conditional_t<FP8, F8Acc<G>, DecAcc<D, G>>;
  constexpr int NH = Acc::NH;
  constexpr int MT = Acc::MT;
  constexpr int KSTEPS = D / 16;
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
  const int gid = lane >> 2, tig = lane & 3;
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
  const int cnt = f0 < f1 ? int(f1 - f0) : 0;
  if (cnt == 0) return;  // no CTA-wide barrier follows

  // offset f -> (sequence, block): the last sequence starting at or before f
  // (empty sequences start where the next one does, so the search passes
  // over them)
  auto locate = [&](long long f, int& s, int& b) {
    int lo = 0, hi = S - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= f) lo = mid;
      else hi = mid - 1;
    }
    s = lo;
    b = int(f - pre[s]);
  };
  // Windows of 32 consecutive pages of the range, lane k holding page
  // 32 w + k: its block id, sequence and block.  The copies run at most
  // kStages pages ahead of the pages being computed, so they stay
  // within the current window (c_) and the next (n_); the one after (p_) is
  // loaded a window ahead, so no page waits on a block-table load.
  int c_id = 0, c_seq = -1, c_blk = 0, n_id = 0, n_seq = -1, n_blk = 0;
  int p_id = 0, p_seq = -1, p_blk = 0;
  auto load_window = [&](int win, int& id, int& sq, int& blk) {
    const long long f = f0 + (long long)win * 32 + lane;
    id = 0;
    sq = -1;
    blk = 0;
    if (f < f1) {
      int ss, b;
      locate(f, ss, b);
      b += first_block_of(p, ss);  // the table's block: after the sequence's prefix
      id = __ldg(p.block_tables + size_t(ss) * p.max_blocks_per_seq + b);
      if (hw == 0 && (id < 0 || id >= p.num_blocks)) atomicOr(&g_decode_error, kErrBadBlockId);
      sq = ss;
      blk = b;
    }
  };
  int wcur = 0;
  load_window(0, c_id, c_seq, c_blk);
  load_window(1, n_id, n_seq, n_blk);
  load_window(2, p_id, p_seq, p_blk);
  // warp-wide: page j of the range (in the current window or the next)
  auto info = [&](int j, int& id, int& sq, int& blk) {
    const bool in_cur = (j >> 5) == wcur;
    id = __shfl_sync(kFull, in_cur ? c_id : n_id, j & 31);
    sq = __shfl_sync(kFull, in_cur ? c_seq : n_seq, j & 31);
    blk = __shfl_sync(kFull, in_cur ? c_blk : n_blk, j & 31);
  };
  // warp-wide: copy page j (KV head hw) into ring stage j % kStages
  // (lane 0 issues)
  auto issue = [&](int j) {
    int id, s, blk;
    info(j, id, s, blk);
    if (lane == 0) {
      const int h = hw;
      // (the decode step has no shared prefix: blocks count from 0)
      if (p.wait_late && blk == pre[s + 1] - pre[s] - 1) {
        griddep_wait();  // the step's append is complete and its rows visible
        if (p.step_slots && h == 0) {
          const int len = __ldg(p.context_lens + s);
          const long long slot = p.step_slots[s];
          const long long want = (long long)id * kBlockTokens + (len - 1) % kBlockTokens;
          if (slot != -1 && slot != want) atomicOr(&g_decode_error, kErrBadSlot);
        }
      }
      const int st = j % kStages;
      const uint32_t bar = bars + st * 8;
      const uint32_t kdst = ring + st * T::kStageBytes;
      const uint32_t vdst = kdst + T::kTileBytes;
      mbar_arrive_expect_tx(bar, T::kStageBytes);
      if constexpr (FP8) {  // one 128-code box per page and tensor
        tma_load_4d(kdst, &tmap_k, bar, 0, h, 0, id);
        tma_load_4d(vdst, &tmap_v, bar, 0, h, 0, id);
      } else {
#pragma unroll
        for (int hh = 0; hh < D / 64; ++hh) {
          tma_load_4d(kdst + hh * T::kHalfBytes, &tmap_k, bar, hh * 64, h, 0, id);
          tma_load_4d(vdst + hh * T::kHalfBytes, &tmap_v, bar, hh * 64, h, 0, id);
        }
      }
    }
  };
  for (int j = 0; j < cnt && j < kStages; ++j) issue(j);
  int issued = cnt < kStages ? cnt : kStages;

  Acc acc;
  uint32_t qf[NH][KSTEPS][2];
  // cur_first / cur_last: the piece's first and last blocks; cur_start /
  // cur_end: the sequence's first own block and one past its last
  int cur_seq = -1, cur_first = 0, cur_last = 0, cur_start = 0, cur_end = 0, cur_len = 0;
  bool cur_extra = false;  // the sequence has a prefix part, merged later
  // the finished piece of (cur_seq, hw): the output when it is the pair's
  // whole context, else its normalised partial at partial slot
  // (cur_seq + g) Hkv + hw (for one head the pieces are ordered by sequence
  // and group alike, so no two share a slot)
  auto flush = [&]() {
#pragma unroll
    for (int nh = 0; nh < NH; ++nh)
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        acc.l[nh][cc] += __shfl_xor_sync(kFull, acc.l[nh][cc], 4);
        acc.l[nh][cc] += __shfl_xor_sync(kFull, acc.l[nh][cc], 8);
        acc.l[nh][cc] += __shfl_xor_sync(kFull, acc.l[nh][cc], 16);
      }
    const int s = cur_seq, h = hw;
    const bool whole = !cur_extra && cur_first == cur_start && cur_last == cur_end - 1;
    const size_t row0 = size_t(s) * p.q_heads + size_t(h) * G;
    const size_t slot = (size_t(s) + size_t(g)) * Hkv + h;
#pragma unroll
    for (int nh = 0; nh < NH; ++nh)
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int head = 8 * nh + 2 * tig + cc;
        if (head >= G) continue;
        const float inv = p.out_scale / acc.l[nh][cc];  // out_scale: the V scale of FP8 pools
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          // the accumulator rows of the m-tile: dims gid and gid + 8 (bf16
          // body), 2 gid and 2 gid + 1 (FP8 body)
          const int dim = FP8 ? 16 * mt + 2 * gid : 16 * mt + gid;
          const int dim2 = FP8 ? dim + 1 : dim + 8;
          const float v0 = acc.o[nh][mt][cc] * inv, v1 = acc.o[nh][mt][cc + 2] * inv;
          if (whole) {
            store_out(p, (row0 + head) * D + dim, v0);
            store_out(p, (row0 + head) * D + dim2, v1);
          } else {
            float* po = p.part_o + (slot * G + head) * D;
            po[dim] = v0;
            po[dim2] = v1;
          }
        }
        if (!whole && gid == 0) p.part_lse[slot * G + head] = acc.m[nh][cc] + __log2f(acc.l[nh][cc]);
      }
  };

  bool failed = false;
  int i = 0;
  while (i < cnt) {
    int id0, seq0, blk0;
    info(i, id0, seq0, blk0);
    bool two = false;
    if (i + 1 < cnt) {
      int id1, seq1, blk1;
      info(i + 1, id1, seq1, blk1);
      two = seq1 == seq0;
    }
    if (seq0 != cur_seq) {
      if (cur_seq >= 0) flush();
      cur_seq = seq0;
      cur_first = blk0;
      const int s = seq0, h = hw;
      cur_start = first_block_of(p, s);
      cur_extra = has_extra(p, s);
      cur_end = cur_start + pre[s + 1] - pre[s];
      const int raw = __ldg(p.context_lens + s);
      cur_len = raw < 0 ? 0 : (raw < cur_end * kBlockTokens ? raw : cur_end * kBlockTokens);
      const size_t row0 = size_t(s) * p.q_heads + size_t(h) * G;
#pragma unroll
      for (int nh = 0; nh < NH; ++nh) {
        const int head = 8 * nh + gid;
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(p.q + (row0 + head) * D);
        if constexpr (FP8) {
          // f16 Q in the FP8 body's k-slot order: dims (4 tig .. 4 tig + 3) of
          // each 16-dim k-step (bf16 -> f16 exact within f16's range)
          bool range_ok = true;
#pragma unroll
          for (int kk = 0; kk < KSTEPS; ++kk) {
            if (head < G) {
              const uint2 wq = __ldg(reinterpret_cast<const uint2*>(
                  p.q + (row0 + head) * D + kk * 16 + 4 * tig));
              qf[nh][kk][0] = bf16x2_to_f16x2(wq.x, &range_ok);
              qf[nh][kk][1] = bf16x2_to_f16x2(wq.y, &range_ok);
            } else {
              qf[nh][kk][0] = qf[nh][kk][1] = 0u;
            }
          }
          if (!range_ok) atomicOr(&g_decode_error, kErrFp16Range);
        } else {
#pragma unroll
          for (int kk = 0; kk < KSTEPS; ++kk) {
            const bool ok = head < G;
            qf[nh][kk][0] = ok ? __ldg(qrow + (kk * 16 + tig * 2) / 2) : 0u;
            qf[nh][kk][1] = ok ? __ldg(qrow + (kk * 16 + 8 + tig * 2) / 2) : 0u;
          }
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
          acc.o[nh][mt][0] = acc.o[nh][mt][1] = acc.o[nh][mt][2] = acc.o[nh][mt][3] = 0.f;
        acc.m[nh][0] = acc.m[nh][1] = -INFINITY;
        acc.l[nh][0] = acc.l[nh][1] = 0.f;
      }
    }
    bool landed = mbar_wait_bounded(bars + (i % kStages) * 8, (i / kStages) & 1);
    if (two && landed)
      landed = mbar_wait_bounded(bars + ((i + 1) % kStages) * 8, ((i + 1) / kStages) & 1);
    if (!__all_sync(kFull, landed)) {
      failed = true;
      break;
    }
    if constexpr (FP8) {
      if (two)
        fp8_pages<G, 2, kStages, 1>(acc, qf, ring, i, blk0 * kBlockTokens, cur_len,
                                    p.scale_log2, lane);
      else
        fp8_pages<G, 1, kStages, 1>(acc, qf, ring, i, blk0 * kBlockTokens, cur_len,
                                    p.scale_log2, lane);
    } else {
      if (two)
        bf16_pages<D, G, 2, 1>(acc, qf, ring, i, blk0 * kBlockTokens, cur_len, p.scale_log2,
                               lane);
      else
        bf16_pages<D, G, 1, 1>(acc, qf, ring, i, blk0 * kBlockTokens, cur_len, p.scale_log2,
                               lane);
    }
    cur_last = blk0 + (two ? 1 : 0);
    __syncwarp();  // every lane is done reading these stages
    const int step = two ? 2 : 1;
    for (int j = i; j < i + step; ++j)
      if (j + kStages < cnt) {
        issue(j + kStages);
        ++issued;
      }
    i += step;
    if ((i >> 5) != wcur && i < cnt) {
      wcur = i >> 5;
      c_id = n_id;
      c_seq = n_seq;
      c_blk = n_blk;
      n_id = p_id;
      n_seq = p_seq;
      n_blk = p_blk;
      load_window(wcur + 2, p_id, p_seq, p_blk);
    }
  }
  if (failed) {
    // Record the timeout and wait (bounded) for this warp's copies still in
    // flight, so no TMA writes into shared memory after the CTA exits.
    if (lane == 0) {
      atomicOr(&g_decode_error, kErrWaitTimeout);
      for (int k = i; k < issued; ++k)
        (void)mbar_wait_bounded(bars + (k % kStages) * 8, (k / kStages) & 1);
    }
    __syncwarp();
    return;
  }
  if (cur_seq >= 0) flush();
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
          flat_chunk(total, flat_groups(fp.total_warps, p.kv_heads), fp.min_pages);
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
