// The per-warp body of the flat split of the paged decode (used by the flat
// decode kernel, paged_decode_flat.cu): one warp streams the pages [f0, f1) of the blocks of all
// sequences laid end to end (sequence s owns offsets pre[s] + b, b < n_s, its
// own blocks after any shared prefix) for one KV head, through its ring of
// page copies, across the sequence boundaries inside the range; it writes a
// pair's output when it holds the pair's whole context and otherwise the
// piece's normalised partial and log2-sum-exp at partial slot (s + g) Hkv +
// h, g the range's index (for one head the pieces are ordered by sequence
// and range alike, so no two share a slot).  bf16 pages take the decode
// body's per-page arithmetic (bf16_pages), FP8 pages the FP8 body's
// (fp8_pages).  Errors go to the including unit's g_decode_error.
#pragma once

#include <climits>
#include <type_traits>

#include "pkv_decode_body.cuh"
#include "pkv_decode_fp8_body.cuh"

namespace pkv {

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
  long long chunk = 0;  // > 0: the blocks per range, given (else from the others)
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

// The flat merge (paged_decode_flat.cu) of the pieces a launch of flat ranges
// wrote, after that launch in the stream.
cudaError_t launch_decode_flat_merge(const DecodeParams& prm, const DecodeFlatParams& fp,
                                     int d_head, cudaStream_t stream);

// A ring stage by page format: bf16 pages (the decode body's 3 stages of one
// 2 x 16 x D x 2-byte page) or FP8 pages (4 stages of 4 KB of e4m3 codes,
// d_head 128).
template <int D, bool FP8>
struct FlatPage {
  static constexpr int kStages = FP8 ? 4 : kDecodeStages;
  static constexpr int kStageBytes = FP8 ? F8Page::kStageBytes : 2 * kBlockTokens * D * 2;
  static constexpr int kTileBytes = kStageBytes / 2;     // K, then V
  static constexpr int kHalfBytes = kBlockTokens * 128;  // a 64-dim bf16 half of a tile
  static constexpr int kRingBytes = kStages * kStageBytes;
};

// One warp's range [f0, f1) in KV head hw, range index g (see above): ring
// and bars are the warp's kStages stages and their mbarriers, initialised
// and with no phase pending.  On return every copy issued has landed (or
// its bounded wait ran out, with PKV_DEVERR_WAIT_TIMEOUT raised).
template <int D, int G, bool FP8>
__device__ __forceinline__ void flat_range(const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                           const DecodeParams& p, const int32_t* pre, int S,
                                           long long f0, long long f1, long long g, int hw,
                                           uint32_t ring, uint32_t bars) {
  using Pg = FlatPage<D, FP8>;
  constexpr int kStages = Pg::kStages;
  using Acc = std::conditional_t<FP8, F8Acc<G>, DecAcc<D, G>>;
  constexpr int NH = Acc::NH;
  constexpr int MT = Acc::MT;
  constexpr int KSTEPS = D / 16;
  constexpr unsigned kFull = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int Hkv = p.kv_heads;
  const int cnt = f0 < f1 ? int(f1 - f0) : 0;
  if (cnt == 0) return;

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
      const uint32_t kdst = ring + st * Pg::kStageBytes;
      const uint32_t vdst = kdst + Pg::kTileBytes;
      mbar_arrive_expect_tx(bar, Pg::kStageBytes);
      if constexpr (FP8) {  // one 128-code box per page and tensor
        tma_load_4d(kdst, &tmap_k, bar, 0, h, 0, id);
        tma_load_4d(vdst, &tmap_v, bar, 0, h, 0, id);
      } else {
#pragma unroll
        for (int hh = 0; hh < D / 64; ++hh) {
          tma_load_4d(kdst + hh * Pg::kHalfBytes, &tmap_k, bar, hh * 64, h, 0, id);
          tma_load_4d(vdst + hh * Pg::kHalfBytes, &tmap_v, bar, hh * 64, h, 0, id);
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


}  // namespace pkv
