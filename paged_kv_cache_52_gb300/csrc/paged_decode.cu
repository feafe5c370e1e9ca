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
//    A warp takes its pages two at a time (two independent chains).
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
#include <climits>
#include <utility>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_decode_common.cuh"

namespace pkv {

static __device__ unsigned g_decode_error = 0;

constexpr int kDecodeWarps = 4;
constexpr int kDecodeStages = 3;
constexpr int kMaxPartitionBlocks = 1024;

int decode_warps_per_cta() { return kDecodeWarps; }

template <int D>
struct DecodeTile {
  static constexpr int kHalfBytes = kBlockTokens * 128;       // 16 rows x 64 bf16
  static constexpr int kTileBytes = kBlockTokens * D * 2;     // one block, one head
  static constexpr int kStageBytes = 2 * kTileBytes;          // K + V
  static constexpr int kRingBytes = kDecodeStages * kStageBytes;
  static constexpr int kRingsBytes = kDecodeWarps * kRingBytes;
  static constexpr int kBarOffset = kRingsBytes;
  static constexpr int kIdsOffset = kBarOffset + kDecodeWarps * kDecodeStages * 8;
  static constexpr int kSmemBytes = kIdsOffset + kMaxPartitionBlocks * 4 + 1024;  // +align slack
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
template <int D, int G, int NP>
__device__ __forceinline__ void bf16_pages(DecAcc<D, G>& A,
                                           const uint32_t (&qf)[(G + 7) / 8][D / 16][2],
                                           uint32_t ring, int i, int tok_first, int len,
                                           float scale_log2, int lane) {
  using T = DecodeTile<D>;
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
    tok0[pg] = tok_first + pg * kDecodeWarps * kBlockTokens;
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
template <int D, int G>
__device__ __forceinline__ void decode_run(const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                           const DecodeParams& p, uint8_t* smem, int seq, int kvh,
                                           int b0, int nb_local, int len, bool final_out,
                                           size_t pbase, int pstride) {
  using T = DecodeTile<D>;
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
  const uint32_t ring = smem_u32(smem + warp * T::kRingBytes);
  const uint32_t bars = smem_u32(smem + T::kBarOffset) + warp * kDecodeStages * 8;
  if (lane == 0) {
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

  const int cnt = warp < nb_local ? (nb_local - warp + kDecodeWarps - 1) / kDecodeWarps : 0;
  auto issue = [&](int i) {
    const int st = i % kDecodeStages;
    const uint32_t bar = bars + st * 8;
    const uint32_t kdst = ring + st * T::kStageBytes;
    const uint32_t vdst = kdst + T::kTileBytes;
    const int bid = ids[warp + i * kDecodeWarps];
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
  // pages two at a time; an odd last page alone
  for (; i < cnt; i += 2) {
    const bool two = i + 1 < cnt;
    bool landed = mbar_wait_bounded(bars + (i % kDecodeStages) * 8, (i / kDecodeStages) & 1);
    if (two && landed)
      landed = mbar_wait_bounded(bars + ((i + 1) % kDecodeStages) * 8,
                                 ((i + 1) / kDecodeStages) & 1);
    if (!__all_sync(0xffffffffu, landed)) {
      failed = true;
      break;
    }
    const int tok_first = (b0 + warp + i * kDecodeWarps) * kBlockTokens;
    if (two)
      bf16_pages<D, G, 2>(acc, qf, ring, i, tok_first, len, p.scale_log2, lane);
    else
      bf16_pages<D, G, 1>(acc, qf, ring, i, tok_first, len, p.scale_log2, lane);

    __syncwarp();  // every lane is done reading these stages
    for (int j = i; j < i + (two ? 2 : 1); ++j) {
      if (j + kDecodeStages < cnt) {
        if (lane == 0) issue(j + kDecodeStages);
        ++issued;
      }
    }
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
  float* mo = reinterpret_cast<float*>(smem + warp * T::kRingBytes);
  float* mml = mo + G * D;
#pragma unroll
  for (int nh = 0; nh < NH; ++nh) {
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
    for (int w = 0; w < kDecodeWarps; ++w) {
      const float* wm = reinterpret_cast<const float*>(smem + w * T::kRingBytes) + G * D;
      big = fmaxf(big, wm[row]);
    }
    float tot = 0.f, val = 0.f;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) {
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

template <int D, int G>
__global__ void __launch_bounds__(kDecodeWarps * 32)
paged_decode_split_kernel(const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_v, const DecodeParams p) {
  griddep_wait();  // inputs may have been written by the previous kernel in the stream
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int pair = blockIdx.x;
  const int part = blockIdx.y;
  const int seq = pair / p.kv_heads;
  const int kvh = pair - seq * p.kv_heads;

  const SeqSpan sp = seq_span(__ldg(p.context_lens + seq), p);
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
  decode_run<D, G>(tmap_k, tmap_v, p, smem, seq, kvh, b0, nb_local, sp.len, final_out,
                   row0 * p.num_parts + part, p.num_parts);
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
constexpr int kListPerThread = kListMaxSeqs / (kDecodeWarps * 32);

template <int D>
struct DecodeListTile {
  static constexpr int kPlanOffset = DecodeTile<D>::kIdsOffset + kMaxPartitionBlocks * 4;
  static constexpr int kSmemBytes = kPlanOffset + (kListMaxSeqs + 1) * 4 + 1024;  // +align slack
};

struct DecodeListParams {
  int32_t* seq_item_base;  // [num_seqs + 1]: first item of each sequence, then the item count
  int num_seqs;            // <= kListMaxSeqs
  int target_items;        // runs aimed at: CTA slots of one wave
  int min_run;             // pages
  int max_blocks;          // page bound per sequence (block table and host max_context_len)
};

// Pages of a sequence in the list plan: its context clamped to max_blocks.
__device__ __forceinline__ int list_pages(int len, int max_blocks) {
  int n = len <= 0 ? 0 : (len + kBlockTokens - 1) / kBlockTokens;
  return n < max_blocks ? n : max_blocks;
}

// Run `item` of the list plan in `base` (every CTA holds the same plan).
template <int D, int G>
__device__ __forceinline__ void list_item(const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                          const DecodeParams& p, const DecodeListParams& lp,
                                          uint8_t* smem, const int32_t* base, int item) {
  constexpr int kThreads = kDecodeWarps * 32;
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
  const int raw_len = __ldg(p.context_lens + seq);
  const int ns = list_pages(raw_len, lp.max_blocks);
  int len = raw_len < 0 ? 0 : raw_len;
  if (len > ns * kBlockTokens) len = ns * kBlockTokens;
  if (len != raw_len && kvh == 0 && run == 0 && threadIdx.x == 0)
    atomicOr(&g_decode_error, kErrBadContext);
  const size_t row0 = size_t(seq) * p.q_heads + size_t(kvh) * G;
  if (ns == 0) {  // empty context: zeros (one run)
    for (int i = threadIdx.x; i < G * D; i += kThreads) store_out(p, row0 * D + i, 0.f);
    return;
  }
  const int b0 = int((long long)run * ns / runs);
  const int b1 = int((long long)(run + 1) * ns / runs);
  decode_run<D, G>(tmap_k, tmap_v, p, smem, seq, kvh, b0, b1 - b0, len, runs == 1,
                   size_t(item) * G, 1);
}

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
  __shared__ long long red_total[kDecodeWarps];
  __shared__ int red_scan[kDecodeWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int S = lp.num_seqs;

  // 1. pages per sequence and their total (thread t owns sequences
  //    t * kListPerThread ..., so the scan below is in sequence order)
  int n[kListPerThread];
  long long mine = 0;
#pragma unroll
  for (int j = 0; j < kListPerThread; ++j) {
    const int s = threadIdx.x * kListPerThread + j;
    n[j] = s < S ? list_pages(__ldg(p.context_lens + s), lp.max_blocks) : 0;
    mine += n[j];
  }
  long long tot = mine;
#pragma unroll
  for (int o = 16; o; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  if (lane == 0) red_total[warp] = tot;
  __syncthreads();
  long long pages = 0;
#pragma unroll
  for (int w = 0; w < kDecodeWarps; ++w) pages += red_total[w];

  // 2. run size and runs per pair.  Rounding k_s up adds at most one run per
  //    pair, so runs of Hkv T / (target - pairs) pages keep the count within
  //    the target (one wave); with fewer slots than pairs every pair has at
  //    least one run anyway.
  const long long pairs = (long long)S * p.kv_heads;
  const long long room = lp.target_items > pairs ? lp.target_items - pairs : lp.target_items;
  long long c = (pages * p.kv_heads + room - 1) / room;
  if (c < lp.min_run) c = lp.min_run;
  if (c > kMaxPartitionBlocks) c = kMaxPartitionBlocks;
  int k[kListPerThread];
  int kmine = 0;
#pragma unroll
  for (int j = 0; j < kListPerThread; ++j) {
    const int s = threadIdx.x * kListPerThread + j;
    k[j] = s < S ? (n[j] > 0 ? int((n[j] + c - 1) / c) : 1) : 0;
    kmine += k[j];
  }

  // 3. exclusive scan of the runs per sequence over the CTA
  int incl = kmine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) red_scan[warp] = incl;
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kDecodeWarps; ++w) {
    before += w < warp ? red_scan[w] : 0;
    all += red_scan[w];
  }
  int run_base = before + incl - kmine;
#pragma unroll
  for (int j = 0; j < kListPerThread; ++j) {
    const int s = threadIdx.x * kListPerThread + j;
    if (s < S) base[s] = run_base * p.kv_heads;
    run_base += k[j];
  }
  if (threadIdx.x == 0) base[S] = all * p.kv_heads;
  __syncthreads();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i <= S; i += kThreads) lp.seq_item_base[i] = base[i];

  // 4. this CTA's items: blockIdx.x, then every gridDim.x-th (a grid smaller
  //    than the item count keeps the decode on at most that many CTAs)
  for (int item = blockIdx.x; item < base[S]; item += gridDim.x) {
    if (item != int(blockIdx.x)) {
      // the previous run is complete: its copies landed and every thread has
      // left its merge; its barriers are retired before they are set up again
      if (lane == 0)
        for (int st = 0; st < kDecodeStages; ++st)
          mbar_inval(smem_u32(smem + DecodeTile<D>::kBarOffset) + (warp * kDecodeStages + st) * 8);
      __syncthreads();
    }
    list_item<D, G>(tmap_k, tmap_v, p, lp, smem, base, item);
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
  if (runs <= 1) return;  // written by the decode kernel
  const size_t r0 = size_t(b + kvh * runs) * G + (h - kvh * G);
  float big = -INFINITY;
  for (int r = 0; r < runs; ++r) big = fmaxf(big, __ldg(p.part_lse + r0 + size_t(r) * G));
  float tot = 0.f;
  float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
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
  const SeqSpan sp = seq_span(__ldg(p.context_lens + seq), p);
  const int nparts_s = span_parts(sp, p);
  const bool extra = p.extra_o != nullptr;
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
  const SeqSpan sp = seq_span(__ldg(p.context_lens + seq), p);
  const int nparts_s = span_parts(sp, p);
  const bool extra = p.extra_o != nullptr;
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

template <int D, int G>
static cudaError_t launch_decode_t(const DecodeParams& prm, int num_seqs,
                                   const CUtensorMap* tmap_k, const CUtensorMap* tmap_v,
                                   cudaStream_t stream) {
  using T = DecodeTile<D>;
  static std::atomic<int> attr_done[kAttrMaxDevices];
  {
    const cudaError_t e =
        set_smem_limit_once(paged_decode_split_kernel<D, G>, T::kSmemBytes, attr_done);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(num_seqs * prm.kv_heads, prm.num_parts);
  cudaError_t e = launch_after_previous(paged_decode_split_kernel<D, G>, grid,
                                        dim3(kDecodeWarps * 32), T::kSmemBytes, stream, *tmap_k,
                                        *tmap_v, prm);
  if (e != cudaSuccess) return e;
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
  const long long rows = (long long)lp.num_seqs * prm.q_heads;
  const long long blocks = (rows * (D / 4) + 255) / 256;
  if (blocks > INT32_MAX) return cudaErrorInvalidValue;
  return launch_after_previous(paged_decode_merge_list_kernel<D>, dim3(unsigned(blocks)),
                               dim3(256), 0, stream, prm, lp, rows);
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
                                   cudaStream_t st) {
  switch (group) {
    case 1: return launch_decode_t<D, 1>(prm, num_seqs, tk, tv, st);
    case 2: return launch_decode_t<D, 2>(prm, num_seqs, tk, tv, st);
    case 4: return launch_decode_t<D, 4>(prm, num_seqs, tk, tv, st);
    case 8: return launch_decode_t<D, 8>(prm, num_seqs, tk, tv, st);
    case 16: return launch_decode_t<D, 16>(prm, num_seqs, tk, tv, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_paged_decode(const DecodeArgs& a, const CUtensorMap* tmap_k,
                                const CUtensorMap* tmap_v, cudaStream_t stream) {
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
  if (a.d_head == 128) return launch_decode_d<128>(prm, a.num_seqs, group, tmap_k, tmap_v, stream);
  if (a.d_head == 64) return launch_decode_d<64>(prm, a.num_seqs, group, tmap_k, tmap_v, stream);
  return cudaErrorInvalidValue;
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
