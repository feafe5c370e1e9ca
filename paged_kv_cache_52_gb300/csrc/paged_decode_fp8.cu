// Paged decode attention over an FP8 (e4m3) KV cache with per-tensor scales.
//
// Same computation as the bf16 decode (paged_decode.cu) on the dequantized
// cache, K = k_scale * e4m3(k_cache), V = v_scale * e4m3(v_cache): the pages
// name FP8 KV caches ("Cache KV, attention et optimisation de l'inference",
// "Utilisez-le": --kv-cache-dtype fp8) as the way to halve decode's KV bytes.
//
// Design (GB300), differences from the bf16 kernel:
//  * a 16-token page of one KV head is 2 KB of codes per tensor: one 4-D TMA
//    box of 128 bytes x 16 rows, 128-byte swizzled; 4 stages per warp, so
//    three CTAs (12 warps) share an SM to hide the longer per-byte compute.
//  * a warp takes its pages two at a time: the two pages' MMA and
//    exponential chains are independent and overlap, and one max reduction,
//    one rescale test and one sum update serve 32 keys.
//  * the contractions run as f16 warp MMAs (m16n8k16, fp32 accumulation):
//    e4m3 -> f16 is exact, bf16 q -> f16 is exact in f16's range (an |q| that
//    would overflow raises PKV_DEVERR_FP16_RANGE), and both scales factor out
//    (k_scale into the softmax scale, v_scale into the output).
//  * the MMAs run transposed, so no MMA row is padding: S^T = K Q^T has the
//    page's 16 keys as M and the group's heads as N (8 per n-tile), O^T = V^T
//    P^T has 16 dims per m-tile as M and the heads as N -- 8 + 8 MMAs per page
//    for a group of 8 instead of 16 + 16 with the heads as (half-empty) M.
//  * K fragments come straight from the code bytes: ldmatrix over the tile as
//    16-bit units hands each thread 4 consecutive dims of a key, which fill the
//    A fragment under a fixed permutation of the 16 dims of a k-step; the Q
//    fragments (B) are loaded with the same permutation, so the dot products
//    are unchanged.
//  * P^T: the S^T accumulator holds (key, two heads) per lane; movmatrix.trans
//    turns each 8 x 8 block into the (two keys, head) layout of the B operand.
//  * V fragments: ldmatrix.trans gives a thread two keys x two adjacent dims;
//    a byte permute splits them into the key pairs of each dim, which are the
//    A fragment rows of an m-tile whose row r is dim 2 r and row r + 8 dim
//    2 r + 1.
//  * P enters PV as one f16 operand: its rounding error is at most 2^-11
//    relative (8x below bf16's), so the output moves by at most 2^-11 times
//    the largest |V| a row attends to; the bf16 kernel needs a hi + lo split
//    for the same bound, this one does not.
#include "pkv_decode_fp8_body.cuh"
#include "pkv_internal.h"

namespace pkv {

static __device__ unsigned g_decode_fp8_error = 0;

constexpr int kF8Warps = 4;
constexpr int kF8Stages = 4;
constexpr int kF8MaxPartitionBlocks = 1024;

struct F8Tile {
  static constexpr int kTileBytes = F8Page::kTileBytes;       // 16 keys x 128 codes
  static constexpr int kStageBytes = F8Page::kStageBytes;     // K + V
  static constexpr int kRingBytes = kF8Stages * kStageBytes;  // 16 KB per warp
  static constexpr int kRingsBytes = kF8Warps * kRingBytes;
  static constexpr int kBarOff = kRingsBytes;
  static constexpr int kIdsOffset = kBarOff + kF8Warps * kF8Stages * 8;
  static constexpr int kSmemBytes = kIdsOffset + kF8MaxPartitionBlocks * 4 + 1024;
};

// The MMAs run transposed: S^T = K Q^T has the 16 keys of a page as its M rows
// and the GQA group's heads as N (8 per n-tile), and O^T = V^T P^T has 16 dims
// per m-tile as M and the heads as N, so no MMA row is padding (with the heads
// as M, a group of 8 fills half of an m16 tile).
template <int G>
__global__ void __launch_bounds__(kF8Warps * 32, 3)
paged_decode_fp8_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const DecodeParams p) {
  griddep_wait();  // inputs may have been written by the previous kernel in the stream
  using T = F8Tile;
  constexpr int D = kF8D;
  constexpr int NH = (G + 7) / 8;  // n-tiles of heads
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  int32_t* ids = reinterpret_cast<int32_t*>(smem + T::kIdsOffset);

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  const int pair = blockIdx.x;
  const int part = blockIdx.y;
  const int seq = pair / p.kv_heads;
  const int kvh = pair - seq * p.kv_heads;

  const SeqSpan sp = seq_span(__ldg(p.context_lens + seq), p, seq);
  const int len = sp.len;
  if (sp.bad && part == 0 && threadIdx.x == 0) atomicOr(&g_decode_fp8_error, kErrBadContext);
  const int nparts_s = span_parts(sp, p);
  if (part >= nparts_s) return;
  const size_t row0 = size_t(seq) * p.q_heads + size_t(kvh) * G;  // first output row
  if (sp.count == 0) {  // empty context: zeros
    for (int i = threadIdx.x; i < G * D; i += blockDim.x) store_out(p, row0 * D + i, 0.f);
    return;
  }
  const int b0 = sp.first + part * p.partition_blocks;  // first block of this partition
  const int nb_local = min(sp.first + sp.count - b0, p.partition_blocks);

  const int32_t* table = p.block_tables + size_t(seq) * p.max_blocks_per_seq + b0;
  for (int i = threadIdx.x; i < nb_local; i += blockDim.x) {
    const int32_t id = __ldg(table + i);
    if (id < 0 || id >= p.num_blocks) atomicOr(&g_decode_fp8_error, kErrBadBlockId);
    ids[i] = id;
  }
  const uint32_t ring = smem_u32(smem + warp * T::kRingBytes);
  const uint32_t bars = smem_u32(smem + T::kBarOff) + warp * kF8Stages * 8;
  if (lane == 0) {
    for (int st = 0; st < kF8Stages; ++st) mbar_init(bars + st * 8, 1);
    fence_barrier_init();
  }
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_v);
  }

  // Q as the B operand of S^T = K Q^T: column n = head gid of n-tile nh, and
  // within the 16 dims of k-step kk the k slots (2 tig, 2 tig + 1) hold dims
  // (4 tig, 4 tig + 1), the slots (2 tig + 8, 2 tig + 9) dims (4 tig + 2,
  // 4 tig + 3) -- the order in which the K fragments arrive (below), so the
  // dot products are unchanged.  Heads past the group are zero.
  uint32_t qf[NH][8][2];
  bool range_ok = true;
#pragma unroll
  for (int nh = 0; nh < NH; ++nh) {
    const int head = 8 * nh + gid;
    const __nv_bfloat16* qrow = p.q + (row0 + head) * D;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      if (head < G) {
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(qrow + kk * 16 + 4 * tig));
        qf[nh][kk][0] = bf16x2_to_f16x2(w.x, &range_ok);
        qf[nh][kk][1] = bf16x2_to_f16x2(w.y, &range_ok);
      } else {
        qf[nh][kk][0] = qf[nh][kk][1] = 0u;
      }
    }
  }
  if (!range_ok) atomicOr(&g_decode_fp8_error, kErrFp16Range);
  __syncthreads();

  const int cnt = warp < nb_local ? (nb_local - warp + kF8Warps - 1) / kF8Warps : 0;
  auto issue = [&](int i) {
    const int st = i % kF8Stages;
    const uint32_t bar = bars + st * 8;
    const uint32_t kdst = ring + st * T::kStageBytes;
    const int bid = ids[warp + i * kF8Warps];
    mbar_arrive_expect_tx(bar, T::kStageBytes);
    tma_load_4d(kdst, &tmap_k, bar, 0, kvh, 0, bid);
    tma_load_4d(kdst + T::kTileBytes, &tmap_v, bar, 0, kvh, 0, bid);
  };
  int issued = 0;
  if (lane == 0) {
    for (int i = 0; i < cnt && i < kF8Stages; ++i) issue(i);
  }
  issued = cnt < kF8Stages ? cnt : kF8Stages;

  F8Acc<G> acc;
#pragma unroll
  for (int nh = 0; nh < F8Acc<G>::NH; ++nh) {
#pragma unroll
    for (int mt = 0; mt < F8Acc<G>::MT; ++mt)
      acc.o[nh][mt][0] = acc.o[nh][mt][1] = acc.o[nh][mt][2] = acc.o[nh][mt][3] = 0.f;
    acc.m[nh][0] = acc.m[nh][1] = -INFINITY;
    acc.l[nh][0] = acc.l[nh][1] = 0.f;
  }
  bool failed = false;
  int i = 0;
  // pages two at a time; an odd last page alone
  for (; i < cnt; i += 2) {
    const bool two = i + 1 < cnt;
    bool landed = mbar_wait_bounded(bars + (i % kF8Stages) * 8, (i / kF8Stages) & 1);
    if (two && landed)
      landed = mbar_wait_bounded(bars + ((i + 1) % kF8Stages) * 8, ((i + 1) / kF8Stages) & 1);
    if (!__all_sync(0xffffffffu, landed)) {
      failed = true;
      break;
    }
    const int tok_first = (b0 + warp + i * kF8Warps) * kBlockTokens;
    if (two)
      fp8_pages<G, 2, kF8Stages, kF8Warps>(acc, qf, ring, i, tok_first, len, p.scale_log2, lane);
    else
      fp8_pages<G, 1, kF8Stages, kF8Warps>(acc, qf, ring, i, tok_first, len, p.scale_log2, lane);

    __syncwarp();
    for (int j = i; j < i + (two ? 2 : 1); ++j) {
      if (j + kF8Stages < cnt) {
        if (lane == 0) issue(j + kF8Stages);
        ++issued;
      }
    }
  }

  if (failed) {
    if (lane == 0) {
      atomicOr(&g_decode_fp8_error, kErrWaitTimeout);
      for (int k = i; k < issued; ++k)
        (void)mbar_wait_bounded(bars + (k % kF8Stages) * 8, (k / kF8Stages) & 1);
    }
    __syncwarp();
  }

#pragma unroll
  for (int nh = 0; nh < F8Acc<G>::NH; ++nh)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      acc.l[nh][c] += __shfl_xor_sync(0xffffffffu, acc.l[nh][c], 4);
      acc.l[nh][c] += __shfl_xor_sync(0xffffffffu, acc.l[nh][c], 8);
      acc.l[nh][c] += __shfl_xor_sync(0xffffffffu, acc.l[nh][c], 16);
    }

  // Cross-warp merge through shared memory ([G][D] partial O, then m, l).
  float* mo = reinterpret_cast<float*>(smem + warp * T::kRingBytes);
  float* mml = mo + G * D;
#pragma unroll
  for (int nh = 0; nh < F8Acc<G>::NH; ++nh) {
    const int h0 = 8 * nh + 2 * tig;
#pragma unroll
    for (int mt = 0; mt < F8Acc<G>::MT; ++mt) {
      const int dim0 = 16 * mt + 2 * gid;
      if (h0 < G) {
        mo[h0 * D + dim0] = acc.o[nh][mt][0];
        mo[h0 * D + dim0 + 1] = acc.o[nh][mt][2];
      }
      if (h0 + 1 < G) {
        mo[(h0 + 1) * D + dim0] = acc.o[nh][mt][1];
        mo[(h0 + 1) * D + dim0 + 1] = acc.o[nh][mt][3];
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

  const bool final_out = (nparts_s == 1) && !p.force_partials;
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int row = idx / D, col = idx - row * D;
    float big = -INFINITY;
#pragma unroll
    for (int w = 0; w < kF8Warps; ++w) {
      const float* wm = reinterpret_cast<const float*>(smem + w * T::kRingBytes) + G * D;
      big = fmaxf(big, wm[row]);
    }
    float tot = 0.f, val = 0.f;
#pragma unroll
    for (int w = 0; w < kF8Warps; ++w) {
      const float* wo = reinterpret_cast<const float*>(smem + w * T::kRingBytes);
      const float wgt = ex2(wo[G * D + row] - big);
      tot += wo[G * D + G + row] * wgt;
      val += wo[row * D + col] * wgt;
    }
    const float res = val / tot * p.out_scale;
    if (final_out) {
      store_out(p, (row0 + row) * D + col, res);
    } else {
      const size_t prow = (row0 + row) * p.num_parts + part;
      p.part_o[prow * D + col] = res;
      if (col == 0) p.part_lse[prow] = big + __log2f(tot);
    }
  }
}

template <int G>
static cudaError_t launch_fp8_t(const DecodeParams& prm, int num_seqs, const CUtensorMap* tk,
                                const CUtensorMap* tv, cudaStream_t stream) {
  static std::atomic<int> attr_done[kAttrMaxDevices];
  {
    const cudaError_t e =
        set_smem_limit_once(paged_decode_fp8_kernel<G>, F8Tile::kSmemBytes, attr_done);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(num_seqs * prm.kv_heads, prm.num_parts);
  cudaError_t e = launch_after_previous(paged_decode_fp8_kernel<G>, grid, dim3(kF8Warps * 32),
                                        F8Tile::kSmemBytes, stream, *tk, *tv, prm);
  if (e != cudaSuccess) return e;
  return launch_decode_merge(prm, num_seqs, kF8D, stream);
}

cudaError_t launch_paged_decode_fp8(const DecodeArgs& a, const CUtensorMap* tmap_k,
                                    const CUtensorMap* tmap_v, cudaStream_t stream) {
  if (a.d_head != kF8D || a.partition_blocks > kF8MaxPartitionBlocks) return cudaErrorInvalidValue;
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
  prm.out_scale = a.out_scale;
  prm.first_block = 0;
  prm.force_partials = 0;
  prm.extra_o = nullptr;
  prm.extra_lse = nullptr;
  prm.out_bf16 = a.out_bf16 ? 1 : 0;
  switch (a.q_heads / a.kv_heads) {
    case 1: return launch_fp8_t<1>(prm, a.num_seqs, tmap_k, tmap_v, stream);
    case 2: return launch_fp8_t<2>(prm, a.num_seqs, tmap_k, tmap_v, stream);
    case 4: return launch_fp8_t<4>(prm, a.num_seqs, tmap_k, tmap_v, stream);
    case 8: return launch_fp8_t<8>(prm, a.num_seqs, tmap_k, tmap_v, stream);
    case 16: return launch_fp8_t<16>(prm, a.num_seqs, tmap_k, tmap_v, stream);
    default: return cudaErrorInvalidValue;
  }
}

// Device address of this unit's error word on the current device.
cudaError_t decode_fp8_error_word(unsigned** word) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(word), g_decode_fp8_error);
}

unsigned read_decode_fp8_error(bool clear) {
  unsigned word = 0;
  if (cudaMemcpyFromSymbol(&word, g_decode_fp8_error, sizeof(word)) != cudaSuccess) return ~0u;
  if (clear) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_decode_fp8_error, &zero, sizeof(zero)) != cudaSuccess) return ~0u;
  }
  return word;
}

}  // namespace pkv
