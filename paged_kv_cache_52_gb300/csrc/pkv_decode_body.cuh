// The bf16 paged-decode body shared by the decode kernels and the fused
// mixed-step kernel: one warp-parallel run over a sequence's pages (TMA rings,
// transposed warp MMAs, online softmax, cross-warp merge) and the
// length-balanced list plan.  Each translation unit that includes this header
// gets its own device error word g_decode_error.
#pragma once

#include <climits>

#include "pkv_decode_common.cuh"
#include "pkv_device.cuh"

namespace pkv {

static __device__ unsigned g_decode_error = 0;

constexpr int kDecodeWarps = 4;   // warps of a decode CTA
constexpr int kDecodeStages = 3;  // ring stages per warp
constexpr int kMaxPartitionBlocks = 1024;

// Shared memory of a run over NW page-owning warps: NW rings of K + V
// stages, their barriers, the run's block ids.
template <int D, int NW>
struct DecodeTile {
  static constexpr int kHalfBytes = kBlockTokens * 128;       // 16 rows x 64 bf16
  static constexpr int kTileBytes = kBlockTokens * D * 2;     // one block, one head
  static constexpr int kStageBytes = 2 * kTileBytes;          // K + V
  static constexpr int kRingBytes = kDecodeStages * kStageBytes;
  static constexpr int kRingsBytes = NW * kRingBytes;
  static constexpr int kBarOffset = kRingsBytes;
  static constexpr int kIdsOffset = kBarOffset + NW * kDecodeStages * 8;
  static constexpr int kEnd = kIdsOffset + kMaxPartitionBlocks * 4;
  static constexpr int kSmemBytes = kEnd + 1024;  // +align slack
};

// An 8x8 matrix of 16-bit values held one row per lane quad (lane l: row
// l / 4, columns 2 (l % 4), 2 (l % 4) + 1) -> the same fragment of its transpose.
__device__ __forceinline__ uint32_t movmatrix_trans_b16(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// Running state of one warp, transposed layout: O^T accumulators (m-tile mt:
// row gid = dim 16 mt + gid, row gid + 8 = dim 16 mt + gid + 8; columns 2 tig,
// 2 tig + 1 = heads 8 nh + 2 tig + c), the running max and this lane's part
// of the row sum of those heads.
template <int D, int G>
struct DecAcc {
  static constexpr int NH = (G + 7) / 8;  // n-tiles of heads
  static constexpr int MT = D / 16;       // m-tiles of dims
  float o[NH][MT][4];
  float m[NH][2], l[NH][2];
};

// NP consecutive landed pages of this warp (ring slots i, i + 1, ...).  The
// MMAs run transposed, so no MMA row is padding: S^T = K Q^T has a page's 16
// keys as M and the group's heads as N (8 per n-tile); O^T = V^T P^T has 16
// dims per m-tile as M and the heads as N -- 8 + 16 MMAs per page for a
// group of 8 (P as hi + lo), where the heads as M (half an m16 tile) took
// 16 + 32.  Two pages per call keep two independent chains in flight and
// share one max reduction and one rescale test among 32 keys.
template <int D, int G, int NP, int NW>
__device__ __forceinline__ void bf16_pages(DecAcc<D, G>& A,
                                           const uint32_t (&qf)[(G + 7) / 8][D / 16][2],
                                           uint32_t ring, int i, int tok_first, int len,
                                           float scale_log2, int lane) {
  using T = DecodeTile<D, NW>;
  constexpr int NH = DecAcc<D, G>::NH;
  constexpr int MT = DecAcc<D, G>::MT;
  constexpr int KSTEPS = D / 16;
  const int gid = lane >> 2, tig = lane & 3;
  const int mi = lane >> 3, mr = lane & 7;
  // K as the A operand (keys x dims): matrices (keys 0-7 | 8-15) x (dims 0-7 | 8-15)
  const int k_key = (mi & 1) * 8 + mr, k_sub = mi >> 1;
  // V^T as the A operand through ldmatrix.trans: matrices (dims 0-7 | 8-15) x (keys 0-7 | 8-15)
  const int v_key = (mi >> 1) * 8 + mr, v_sub = mi & 1;
  uint32_t kbase[NP];
  int tok0[NP];
#pragma unroll
  for (int pg = 0; pg < NP; ++pg) {
    kbase[pg] = ring + ((i + pg) % kDecodeStages) * T::kStageBytes;
    tok0[pg] = tok_first + pg * NW * kBlockTokens;
  }

  // S^T = K Q^T; even and odd k-steps accumulate separately (shorter chains).
  float s[NP][NH][4], s_odd[NP][NH][4];
#pragma unroll
  for (int pg = 0; pg < NP; ++pg)
#pragma unroll
    for (int nh = 0; nh < NH; ++nh)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[pg][nh][e] = s_odd[pg][nh][e] = 0.f;
#pragma unroll
  for (int kk = 0; kk < KSTEPS; ++kk) {
#pragma unroll
    for (int pg = 0; pg < NP; ++pg) {
      const int chunk = 2 * kk + k_sub;
      uint32_t a0, a1, a2, a3;
      ldsm_x4(kbase[pg] + (chunk >> 3) * T::kHalfBytes + k_key * 128 +
                  (((chunk & 7) ^ (k_key & 7)) << 4),
              a0, a1, a2, a3);
#pragma unroll
      for (int nh = 0; nh < NH; ++nh)
        mma_bf16_16816((kk & 1) ? s_odd[pg][nh] : s[pg][nh], a0, a1, a2, a3, qf[nh][kk][0],
                       qf[nh][kk][1]);
    }
  }

  // Online softmax in the log2 domain per head column over the pages' keys
  // (rows gid and gid + 8 of each page here; the other keys in the lanes with
  // the same tig).  Keys at or past the length are excluded.
  bool k0_in[NP], k1_in[NP];
#pragma unroll
  for (int pg = 0; pg < NP; ++pg) {
    k0_in[pg] = tok0[pg] + gid < len;
    k1_in[pg] = tok0[pg] + gid + 8 < len;
  }
  uint32_t ph[NP][NH][2], pl[NP][NH][2];  // P^T (B operand) hi and lo: keys 2 tig.., 8 + 2 tig..
  bool all_same = true;
  float alpha[NH][2];
#pragma unroll
  for (int nh = 0; nh < NH; ++nh) {
    float pr[NP][4];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float x0[NP], x1[NP];
      float mx = -INFINITY;
#pragma unroll
      for (int pg = 0; pg < NP; ++pg) {
        x0[pg] = k0_in[pg] ? (s[pg][nh][c] + s_odd[pg][nh][c]) * scale_log2 : -INFINITY;
        x1[pg] = k1_in[pg] ? (s[pg][nh][c + 2] + s_odd[pg][nh][c + 2]) * scale_log2 : -INFINITY;
        mx = fmaxf(mx, fmaxf(x0[pg], x1[pg]));
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float mn = fmaxf(A.m[nh][c], mx);
      alpha[nh][c] = ex2(A.m[nh][c] - mn);
      all_same = all_same && A.m[nh][c] == mn;
      A.m[nh][c] = mn;
      float add = 0.f;
#pragma unroll
      for (int pg = 0; pg < NP; ++pg) {
        pr[pg][c] = ex2(x0[pg] - mn);
        pr[pg][c + 2] = ex2(x1[pg] - mn);
        add += pr[pg][c] + pr[pg][c + 2];
      }
      A.l[nh][c] = A.l[nh][c] * alpha[nh][c] + add;
    }
    // P^T: the lane's (key, two heads) pairs as bf16 hi and the bf16
    // residual lo, each 8 x 8 block transposed into (two keys, head)
#pragma unroll
    for (int pg = 0; pg < NP; ++pg)
#pragma unroll
      for (int r = 0; r < 2; ++r) {  // keys gid (r = 0) / gid + 8 (r = 1)
        const uint32_t h = pack_bf16x2(pr[pg][2 * r], pr[pg][2 * r + 1]);
        const uint32_t l = pack_bf16x2(pr[pg][2 * r] - bf16_lo_to_f32(h),
                                       pr[pg][2 * r + 1] - bf16_hi_to_f32(h));
        ph[pg][nh][r] = movmatrix_trans_b16(h);
        pl[pg][nh][r] = movmatrix_trans_b16(l);
      }
  }
  // After the first pages the running max rarely moves: skip the rescale
  // (alpha = 1 exactly, so the result is unchanged) unless some head needs it.
  if (!__all_sync(0xffffffffu, all_same)) {
#pragma unroll
    for (int nh = 0; nh < NH; ++nh)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        A.o[nh][mt][0] *= alpha[nh][0];
        A.o[nh][mt][1] *= alpha[nh][1];
        A.o[nh][mt][2] *= alpha[nh][0];
        A.o[nh][mt][3] *= alpha[nh][1];
      }
  }

  // Rows of the last page past the length may hold anything, NaN included;
  // their P is 0, and zeroing their V keeps each such product exactly 0.  A
  // V^T register holds keys (2 tig, 2 tig + 1) -- or 8 more -- in its halves.
  uint32_t vm0[NP], vm1[NP];
#pragma unroll
  for (int pg = 0; pg < NP; ++pg) {
    vm0[pg] = vm1[pg] = 0xffffffffu;
    if (tok0[pg] + kBlockTokens > len) {
      const int k0 = tok0[pg] + 2 * tig;
      vm0[pg] = (k0 < len ? 0x0000ffffu : 0u) | (k0 + 1 < len ? 0xffff0000u : 0u);
      vm1[pg] = (k0 + 8 < len ? 0x0000ffffu : 0u) | (k0 + 9 < len ? 0xffff0000u : 0u);
    }
  }
  // O^T += V^T P^T: one ldmatrix.trans per 16-dim m-tile and page; the hi
  // products of all m-tiles first, then the lo ones, so no two consecutive
  // MMAs share an accumulator.
  uint32_t va[NP][MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int pg = 0; pg < NP; ++pg) {
      const int chunk = 2 * mt + v_sub;
      ldsm_x4_trans(kbase[pg] + T::kTileBytes + (chunk >> 3) * T::kHalfBytes + v_key * 128 +
                        (((chunk & 7) ^ (v_key & 7)) << 4),
                    va[pg][mt][0], va[pg][mt][1], va[pg][mt][2], va[pg][mt][3]);
      va[pg][mt][0] &= vm0[pg];
      va[pg][mt][1] &= vm0[pg];
      va[pg][mt][2] &= vm1[pg];
      va[pg][mt][3] &= vm1[pg];
    }
#pragma unroll
  for (int pg = 0; pg < NP; ++pg)
#pragma unroll
    for (int nh = 0; nh < NH; ++nh)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
        mma_bf16_16816(A.o[nh][mt], va[pg][mt][0], va[pg][mt][1], va[pg][mt][2], va[pg][mt][3],
                       ph[pg][nh][0], ph[pg][nh][1]);
#pragma unroll
  for (int pg = 0; pg < NP; ++pg)
#pragma unroll
    for (int nh = 0; nh < NH; ++nh)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
        mma_bf16_16816(A.o[nh][mt], va[pg][mt][0], va[pg][mt][1], va[pg][mt][2], va[pg][mt][3],
                       pl[pg][nh][0], pl[pg][nh][1]);
}

// One run of `nb_local` pages of sequence `seq`, KV head `kvh`, starting at
// block b0, for the G query heads of the group: softmax(q K^T * scale) V over
// the run's keys below `len`.  final_out: the run is the sequence's whole
// context and writes the output; otherwise it writes its normalised partial
// output and log2-sum-exp at partial row pbase + head * pstride.
// PAIR: a warp takes its pages two at a time (two independent MMA and
// exponential chains; its ring is refilled after both), else one at a time
// (each stage refilled as soon as its page is done: more bytes in flight).
template <int D, int G, int NW, bool PAIR = true>
__device__ __forceinline__ void decode_run(const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                           const DecodeParams& p, uint8_t* smem, int seq, int kvh,
                                           int b0, int nb_local, int len, bool final_out,
                                           size_t pbase, int pstride) {
  using T = DecodeTile<D, NW>;
  using Acc = DecAcc<D, G>;
  constexpr int NH = Acc::NH;
  constexpr int MT = Acc::MT;
  constexpr int KSTEPS = D / 16;
  int32_t* ids = reinterpret_cast<int32_t*>(smem + T::kIdsOffset);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  const size_t row0 = size_t(seq) * p.q_heads + size_t(kvh) * G;  // first output row

  // Stage this partition's block ids; ids outside the pool are flagged (their
  // TMA boxes are out of bounds and read as zeros).
  const int32_t* table = p.block_tables + size_t(seq) * p.max_blocks_per_seq + b0;
  for (int i = threadIdx.x; i < nb_local; i += blockDim.x) {
    const int32_t id = __ldg(table + i);
    if (id < 0 || id >= p.num_blocks) atomicOr(&g_decode_error, kErrBadBlockId);
    ids[i] = id;
  }
  // Warps from NW on own no ring: they only help stage the ids and write the
  // output (a CTA whose other warps have other roles).
  const bool pager = warp < NW;
  const uint32_t ring = smem_u32(smem + (pager ? warp : 0) * T::kRingBytes);
  const uint32_t bars = smem_u32(smem + T::kBarOffset) + (pager ? warp : 0) * kDecodeStages * 8;
  if (pager && lane == 0) {
    for (int st = 0; st < kDecodeStages; ++st) mbar_init(bars + st * 8, 1);
    fence_barrier_init();
  }
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_v);
  }

  // Q as the B operand of S^T = K Q^T: column gid of n-tile nh = head
  // 8 nh + gid (zero past the group), k slots (2 tig, 2 tig + 1) and
  // (2 tig + 8, 2 tig + 9) = those dims of the 16-dim k-step.
  uint32_t qf[NH][KSTEPS][2];
#pragma unroll
  for (int nh = 0; nh < NH; ++nh) {
    const int head = 8 * nh + gid;
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(p.q + (row0 + head) * D);
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      const bool ok = head < G;
      qf[nh][kk][0] = ok ? __ldg(qrow + (kk * 16 + tig * 2) / 2) : 0u;
      qf[nh][kk][1] = ok ? __ldg(qrow + (kk * 16 + 8 + tig * 2) / 2) : 0u;
    }
  }
  __syncthreads();  // ids staged, barriers initialised

  const int cnt = (pager && warp < nb_local) ? (nb_local - warp + NW - 1) / NW : 0;
  // the page holding the sequence's last position (the step's appended
  // token when the append runs beside this grid: its loads wait for it)
  const int last_page = len > 0 ? (len - 1) / kBlockTokens : -1;
  auto issue = [&](int i) {
    const int st = i % kDecodeStages;
    const uint32_t bar = bars + st * 8;
    const uint32_t kdst = ring + st * T::kStageBytes;
    const uint32_t vdst = kdst + T::kTileBytes;
    const int bid = ids[warp + i * NW];
    if (p.wait_late && b0 + warp + i * NW == last_page) {
      griddep_wait();  // the append is complete and its rows are visible
      if (p.step_slots && kvh == 0) {
        // the append must have written exactly this position (or skipped it)
        const long long slot = p.step_slots[seq];
        const long long want = (long long)bid * kBlockTokens + (len - 1) % kBlockTokens;
        if (slot != -1 && slot != want) atomicOr(&g_decode_error, kErrBadSlot);
      }
    }
    mbar_arrive_expect_tx(bar, T::kStageBytes);
#pragma unroll
    for (int h = 0; h < D / 64; ++h) {
      tma_load_4d(kdst + h * T::kHalfBytes, &tmap_k, bar, h * 64, kvh, 0, bid);
      tma_load_4d(vdst + h * T::kHalfBytes, &tmap_v, bar, h * 64, kvh, 0, bid);
    }
  };
  int issued = 0;
  if (lane == 0) {
    for (int i = 0; i < cnt && i < kDecodeStages; ++i) issue(i);
  }
  issued = cnt < kDecodeStages ? cnt : kDecodeStages;

  Acc acc;
#pragma unroll
  for (int nh = 0; nh < NH; ++nh) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
      acc.o[nh][mt][0] = acc.o[nh][mt][1] = acc.o[nh][mt][2] = acc.o[nh][mt][3] = 0.f;
    acc.m[nh][0] = acc.m[nh][1] = -INFINITY;
    acc.l[nh][0] = acc.l[nh][1] = 0.f;
  }
  bool failed = false;
  int i = 0;
  // pages two at a time (PAIR) with an odd last page alone, or one at a time
  for (; i < cnt;) {
    const bool two = PAIR && i + 1 < cnt;
    bool landed = mbar_wait_bounded(bars + (i % kDecodeStages) * 8, (i / kDecodeStages) & 1);
    if (two && landed)
      landed = mbar_wait_bounded(bars + ((i + 1) % kDecodeStages) * 8,
                                 ((i + 1) / kDecodeStages) & 1);
    if (!__all_sync(0xffffffffu, landed)) {
      failed = true;
      break;
    }
    const int tok_first = (b0 + warp + i * NW) * kBlockTokens;
    if (two)
      bf16_pages<D, G, 2, NW>(acc, qf, ring, i, tok_first, len, p.scale_log2, lane);
    else
      bf16_pages<D, G, 1, NW>(acc, qf, ring, i, tok_first, len, p.scale_log2, lane);

    __syncwarp();  // every lane is done reading these stages
    for (int j = i; j < i + (two ? 2 : 1); ++j) {
      if (j + kDecodeStages < cnt) {
        if (lane == 0) issue(j + kDecodeStages);
        ++issued;
      }
    }
    i += two ? 2 : 1;
  }

  if (failed) {
    // Record the timeout and wait (bounded) for this warp's copies still in
    // flight, so no TMA writes into shared memory after the CTA exits.
    if (lane == 0) {
      atomicOr(&g_decode_error, kErrWaitTimeout);
      for (int k = i; k < issued; ++k)
        (void)mbar_wait_bounded(bars + (k % kDecodeStages) * 8, (k / kDecodeStages) & 1);
    }
    __syncwarp();
  }

  // Row sums were kept per lane: reduce over the lanes of one head column.
#pragma unroll
  for (int nh = 0; nh < NH; ++nh)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      acc.l[nh][c] += __shfl_xor_sync(0xffffffffu, acc.l[nh][c], 4);
      acc.l[nh][c] += __shfl_xor_sync(0xffffffffu, acc.l[nh][c], 8);
      acc.l[nh][c] += __shfl_xor_sync(0xffffffffu, acc.l[nh][c], 16);
    }

  // Cross-warp merge through shared memory (each warp reuses its own ring):
  // [G][D] partial O, then m[G], l[G].
  float* mo = reinterpret_cast<float*>(smem + (pager ? warp : 0) * T::kRingBytes);
  float* mml = mo + G * D;
#pragma unroll
  for (int nh = 0; nh < NH; ++nh) {
    if (!pager) break;
    const int h0 = 8 * nh + 2 * tig;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int dim = 16 * mt + gid;
      if (h0 < G) {
        mo[h0 * D + dim] = acc.o[nh][mt][0];
        mo[h0 * D + dim + 8] = acc.o[nh][mt][2];
      }
      if (h0 + 1 < G) {
        mo[(h0 + 1) * D + dim] = acc.o[nh][mt][1];
        mo[(h0 + 1) * D + dim + 8] = acc.o[nh][mt][3];
      }
    }
    if (gid == 0) {
#pragma unroll
      for (int c = 0; c < 2; ++c)
        if (h0 + c < G) {
          mml[h0 + c] = acc.m[nh][c];
          mml[G + h0 + c] = acc.l[nh][c];
        }
    }
  }
  __syncthreads();

  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int row = idx / D, col = idx - row * D;
    float big = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float* wm = reinterpret_cast<const float*>(smem + w * T::kRingBytes) + G * D;
      big = fmaxf(big, wm[row]);
    }
    float tot = 0.f, val = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float* wo = reinterpret_cast<const float*>(smem + w * T::kRingBytes);
      const float wgt = ex2(wo[G * D + row] - big);
      tot += wo[G * D + G + row] * wgt;
      val += wo[row * D + col] * wgt;
    }
    const float res = val / tot;
    if (final_out) {
      store_out(p, (row0 + row) * D + col, res);
    } else {
      const size_t prow = pbase + size_t(row) * pstride;
      p.part_o[prow * D + col] = res;
      if (col == 0) p.part_lse[prow] = big + __log2f(tot);
    }
  }
}

// ---------------------------------------------------------------------------
// Length-balanced work list.  With fewer (sequence, KV head) pairs than CTA
// slots, uniform partitions sized from the longest context leave the waves
// unbalanced: how the real lengths fall into partitions decides the tail.
// Here every CTA derives the same plan from the context lengths on the device:
//   n_s  pages of sequence s (clamped to the block table and the host bound),
//   T    = sum_s n_s,
//   c    = clamp(ceil(Hkv T / (target - pairs)), min_run, kMaxPartitionBlocks)
//          pages (target alone when it is not above the pair count),
//   k_s  = max(1, ceil(n_s / c)) runs per (s, KV head), of near-equal size
//          (run r covers blocks [r n_s / k_s, (r + 1) n_s / k_s)),
// items numbered sequence-major, then KV head, then run; CTA i takes item i
// (and every gridDim.x-th after it on a smaller grid).  Every run is at most
// c pages and, when the target exceeds the pair count, there are at most
// `target` of them, so a grid of `target` CTA slots finishes in one even
// wave.  A pair with one run writes the output; otherwise its runs write
// partials at rows item * G + head and the list merge combines them.
// Block 0 stores the per-sequence first items (seq_item_base) for the merge.
// ---------------------------------------------------------------------------
constexpr int kListMaxSeqs = 512;

template <int D>
struct DecodeListTile {
  static constexpr int kPlanOffset = DecodeTile<D, kDecodeWarps>::kIdsOffset + kMaxPartitionBlocks * 4;
  static constexpr int kSmemBytes = kPlanOffset + (kListMaxSeqs + 1) * 4 + 1024;  // +align slack
};

// The list plan of S <= kListMaxSeqs sequences, computed by all NT threads of
// a block: base[s] = the first run of sequence s (its KV heads' runs are
// consecutive), base[S] = the run count.  The run size c is the smallest in
// [max(min_run, ceil(Hkv T / target)), kMaxPartitionBlocks] for which the
// runs fit the target (binary search over the block-wide run count); when
// none fits (more pairs than the target, or runs capped at
// kMaxPartitionBlocks pages) the largest is taken.
template <int NT>
__device__ void list_plan(const DecodeParams& p, const DecodeListParams& lp, int32_t* base) {
  constexpr int PER = (kListMaxSeqs + NT - 1) / NT;
  constexpr int NWARPS = NT / 32;
  __shared__ long long red_ll[NWARPS];
  __shared__ int red_i[NWARPS];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int S = lp.num_seqs;
  auto block_sum = [&](long long v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();  // the previous use of red_ll is over
    if (lane == 0) red_ll[warp] = v;
    __syncthreads();
    long long t = 0;
#pragma unroll
    for (int w = 0; w < NWARPS; ++w) t += red_ll[w];
    return t;
  };
  // pages of this thread's sequences (thread t owns t * PER ..., in order)
  int n[PER];
  long long mine = 0, top = 0;
  bool pre[PER];  // the sequence merges a shared-prefix partial
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int s = threadIdx.x * PER + j;
    int f = 0;
    n[j] = s < S ? list_own_pages(p, lp, s, &f) : 0;
    pre[j] = f > 0 && p.extra_o != nullptr;
    mine += n[j];
    top = n[j] > top ? n[j] : top;
  }
  const long long pages = block_sum(mine);
  long long mx = top;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const long long v = __shfl_xor_sync(0xffffffffu, mx, o);
    mx = v > mx ? v : mx;
  }
  __syncthreads();
  if (lane == 0) red_ll[warp] = mx;
  __syncthreads();
  long long longest = 0;
#pragma unroll
  for (int w = 0; w < NWARPS; ++w) longest = red_ll[w] > longest ? red_ll[w] : longest;
  // runs at run size c, over the block
  // runs of a sequence: its own pages cut at c; an empty one still takes a
  // run (it writes zeros) unless a prefix partial carries its whole result
  auto runs_of = [&](int j, int c) { return n[j] > 0 ? (n[j] + c - 1) / c : (pre[j] ? 0 : 1); };
  auto runs_at = [&](int c) {
    long long r = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j)
      if (threadIdx.x * PER + j < S) r += runs_of(j, c);
    return block_sum(r) * p.kv_heads;
  };
  long long lo = (pages * p.kv_heads + lp.target_items - 1) / lp.target_items;
  if (lo < lp.min_run) lo = lp.min_run;
  long long hi = longest < kMaxPartitionBlocks ? longest : kMaxPartitionBlocks;
  if (lo > hi) lo = hi;
  if (lo < 1) lo = hi = 1;
  int c = int(hi);
  if (runs_at(int(hi)) <= lp.target_items) {
    while (lo < hi) {  // uniform over the block: every thread takes the same branch
      const long long mid = (lo + hi) / 2;
      if (runs_at(int(mid)) <= lp.target_items) hi = mid;
      else lo = mid + 1;
    }
    c = int(lo);
  }
  // exclusive scan of the runs per sequence
  int k[PER];
  int kmine = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int s = threadIdx.x * PER + j;
    k[j] = s < S ? runs_of(j, c) : 0;
    kmine += k[j];
  }
  int incl = kmine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  __syncthreads();
  if (lane == 31) red_i[warp] = incl;
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < NWARPS; ++w) {
    before += w < warp ? red_i[w] : 0;
    all += red_i[w];
  }
  int run_base = before + incl - kmine;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int s = threadIdx.x * PER + j;
    if (s < S) base[s] = run_base * p.kv_heads;
    run_base += k[j];
  }
  if (threadIdx.x == 0) base[S] = all * p.kv_heads;
  __syncthreads();
}

// Run `item` of the list plan in `base` (every CTA holds the same plan).
template <int D, int G, int NW, bool PAIR = true>
__device__ __forceinline__ void list_item(const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                          const DecodeParams& p, const DecodeListParams& lp,
                                          uint8_t* smem, const int32_t* base, int item) {
  const int S = lp.num_seqs;
  int lo = 0, hi = S - 1;  // the last sequence whose first item is <= item
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (base[mid] <= item) lo = mid;
    else hi = mid - 1;
  }
  const int seq = lo;
  const int runs = (base[seq + 1] - base[seq]) / p.kv_heads;
  const int local = item - base[seq];
  const int kvh = local / runs;
  const int run = local - kvh * runs;
  const int raw_len = p.context_lens[seq];
  int first = 0;
  const int ns = list_own_pages(p, lp, seq, &first);  // pages after the shared prefix
  const int end = (first + ns) * kBlockTokens;
  int len = raw_len < 0 ? 0 : raw_len;
  if (len > end) len = end;
  if (len != raw_len && kvh == 0 && run == 0 && threadIdx.x == 0)
    atomicOr(&g_decode_error, kErrBadContext);
  const size_t row0 = size_t(seq) * p.q_heads + size_t(kvh) * G;
  if (ns == 0) {  // empty context: zeros (one run; a prefix partial takes no run)
    for (int i = threadIdx.x; i < G * D; i += blockDim.x) store_out(p, row0 * D + i, 0.f);
    return;
  }
  const int b0 = first + int((long long)run * ns / runs);
  const int b1 = first + int((long long)(run + 1) * ns / runs);
  // a sequence with a prefix partial always leaves its runs to the merge
  const bool final_out = runs == 1 && !has_extra(p, seq);
  decode_run<D, G, NW, PAIR>(tmap_k, tmap_v, p, smem, seq, kvh, b0, b1 - b0, len, final_out,
                             size_t(item) * G, 1);
}

}  // namespace pkv
