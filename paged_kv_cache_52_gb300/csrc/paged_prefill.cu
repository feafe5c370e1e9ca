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
//  * one CTA per (128-row query tile, sequence x KV head).  The 128 rows are
//    128/G query tokens x the G heads of the GQA group (rows token-major), so
//    one TMA box brings the tile in and every K/V tile serves all G heads.
//    Tiles are launched longest-first (the last tiles of a chunk see the most
//    keys).
//  * warp roles: warps 0-3 softmax / correction / epilogue (thread = row =
//    TMEM lane), warp 4 TMA producer (32 lanes issue the 32 per-block boxes
//    of a K+V tile), warp 5 MMA issuer (one thread).
//  * S = Q K^T (M=128, N=128, K=d) into one of two TMEM S buffers; the MMA
//    warp issues S for tile j+2 while softmax works on tile j+1, then
//    O += P V (M=128, N=d, K=128) into a TMEM O accumulator.  Q, K, P are
//    K-major 128-byte-swizzled operands; V is the MN-major operand straight
//    from the pool layout, so no transpose pass is needed.
//  * P enters the PV product as bf16 hi + bf16 lo (two MMAs per k-step), so
//    its rounding error is ~2^-17 relative instead of bf16's 2^-9 -- needed
//    for rows that see only a few keys, where one rounded weight moves the
//    output by more than 2e-3.
//  * online softmax in base 2 with lazy rescaling: the running max used for
//    the exponentials only moves when a row's new max exceeds it by more than
//    8 (a factor 256), and only then is that row's O rescaled in TMEM.  The
//    final division uses the same stale max for O and the row sum, so the
//    result is exact in real arithmetic.
//  * every mbarrier wait is bounded; a timeout sets an error bit and an abort
//    flag that the other roles see, copies and MMAs in flight are drained
//    (bounded) and tensor memory is freed before the CTA exits.
#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_tcgen05.cuh"

namespace pkv {

static __device__ unsigned g_prefill_error = 0;

constexpr int kPfRows = 128;          // query rows per CTA (tokens x heads)
constexpr int kPfKvTile = 128;        // keys per K/V tile (8 pages of 16)
constexpr int kPfStages = 2;          // K/V tile ring
constexpr int kPfThreads = 192;       // 4 softmax warps + TMA warp + MMA warp
constexpr int kPfProducerWarp = 4;
constexpr int kPfMmaWarp = 5;
constexpr uint32_t kPfTmemCols = 512; // S0 | S1 | O
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows by > x256

template <int D>
struct PrefillSmem {
  static constexpr int kHalf = kPfRows * 128;                // 128 rows x 64 bf16 (16 KB)
  static constexpr int kQBytes = (D / 64) * kHalf;
  static constexpr int kTileBytes = (D / 64) * kHalf;        // K or V: 128 keys x D
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kPBytes = 2 * kHalf;                  // P: 128 rows x 128 keys bf16
  static constexpr int kQOff = 0;
  static constexpr int kStageOff = kQOff + kQBytes;
  static constexpr int kPOff = kStageOff + kPfStages * kStageBytes;  // P hi, then P lo
  static constexpr int kBarOff = kPOff + 2 * kPBytes;
  // q_full, kv_full[2], kv_empty[2], s_full[2], p_full, o_done, drain
  static constexpr int kNumBars = 10;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;     // tmem base, abort flag
  static constexpr int kUsed = kMiscOff + 16 + 1024;          // + alignment slack
  // One CTA per SM: it holds all 512 TMEM columns.
  static constexpr int kSmemBytes = kUsed > 120 * 1024 ? kUsed : 120 * 1024;
  static_assert(kSmemBytes <= 232448, "prefill tile does not fit in shared memory");
};

enum PfBar { kQFull = 0, kKvFull0 = 1, kKvEmpty0 = 3, kSFull0 = 5, kPFull = 7, kODone = 8,
             kDrain = 9 };

struct PrefillParams {
  const int32_t* q_start;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* out;
  int num_seqs, q_heads, kv_heads, num_blocks, max_blocks_per_seq, total_q, max_q_len;
  int causal;
  float scale_log2;
};

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool pf_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  for (uint32_t i = 0; i < kWaitPollLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u && *abort_flag) return false;
  }
  return false;
}

__device__ __forceinline__ void pf_abort(volatile int* abort_flag) {
  *abort_flag = 1;
  atomicOr(&g_prefill_error, kErrWaitTimeout);
}

template <int D, int G>
__global__ void __launch_bounds__(kPfThreads, 1)
paged_prefill_kernel(const __grid_constant__ CUtensorMap tmap_q,
                     const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const PrefillParams p) {
  using L = PrefillSmem<D>;
  constexpr int TPT = kPfRows / G;  // query tokens per tile
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + L::kBarOff;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = blockIdx.y;
  const int seq = pair / p.kv_heads;
  const int kvh = pair - seq * p.kv_heads;
  const int tile = int(gridDim.x) - 1 - int(blockIdx.x);  // longest-first

  // ---- per-CTA bounds (uniform over the CTA, so early exits are safe)
  const int qs = __ldg(p.q_start + seq), qe = __ldg(p.q_start + seq + 1);
  const int ctx = __ldg(p.context_lens + seq);
  const int n = qe - qs;
  if (qs < 0 || n < 0 || qe > p.total_q || n > ctx ||
      ctx > p.max_blocks_per_seq * 16) {
    if (tile == 0 && threadIdx.x == 0) atomicOr(&g_prefill_error, kErrBadQueryRange);
    return;
  }
  if (n > p.max_q_len && tile == 0 && threadIdx.x == 0)
    atomicOr(&g_prefill_error, kErrBadQueryRange);  // tiles past the grid are not computed
  const int t0 = tile * TPT;
  if (t0 >= n) return;
  const int tok_valid = min(TPT, n - t0);
  const int kv_end = p.causal ? (ctx - n + t0 + tok_valid) : ctx;  // keys [0, kv_end)
  const int ntiles = (kv_end + kPfKvTile - 1) / kPfKvTile;
  const int nblk = (ctx + 15) / 16;

  // ---- set-up: barriers (producer lane 0), tensor memory (warp 0)
  if (warp == kPfProducerWarp && lane == 0) {
    mbar_init(bars + 8 * kQFull, 1);
    for (int s = 0; s < kPfStages; ++s) {
      mbar_init(bars + 8 * (kKvFull0 + s), 1);
      mbar_init(bars + 8 * (kKvEmpty0 + s), 1);
      mbar_init(bars + 8 * (kSFull0 + s), 1);
    }
    mbar_init(bars + 8 * kPFull, 4);
    mbar_init(bars + 8 * kODone, 1);
    mbar_init(bars + 8 * kDrain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kPfTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t q_smem = sbase + L::kQOff;
  const uint32_t p_smem = sbase + L::kPOff;

  if (warp == kPfProducerWarp) {
    // ================= TMA producer =================
    int issued_q = 0, issued[kPfStages] = {0, 0};
    if (lane == 0) {
      tma_prefetch_desc(&tmap_q);
      tma_prefetch_desc(&tmap_k);
      tma_prefetch_desc(&tmap_v);
      mbar_arrive_expect_tx(bars + 8 * kQFull, L::kQBytes);
#pragma unroll
      for (int h = 0; h < D / 64; ++h)
        tma_load_3d(q_smem + h * L::kHalf, &tmap_q, bars + 8 * kQFull, h * 64, kvh * G, qs + t0);
      issued_q = 1;
    }
    const int32_t* table = p.block_tables + size_t(seq) * p.max_blocks_per_seq;
    constexpr int kLoads = 2 * 8 * (D / 64);  // K and V, 8 pages, D/64 column halves
    for (int j = 0; j < ntiles; ++j) {
      const int st = j % kPfStages;
      if (j >= kPfStages) {
        const bool ok = __all_sync(0xffffffffu,
                                   pf_wait(bars + 8 * (kKvEmpty0 + st), ((j / kPfStages) - 1) & 1,
                                           abort_flag));
        if (!ok) {
          if (lane == 0) pf_abort(abort_flag);
          break;
        }
      }
      if (lane == 0) mbar_arrive_expect_tx(bars + 8 * (kKvFull0 + st), L::kStageBytes);
      __syncwarp();
      if (lane < kLoads) {
        const int kv = lane / (8 * (D / 64));
        const int b = (lane / (D / 64)) & 7;
        const int h = lane % (D / 64);
        const int blk = j * 8 + b;
        int id = -1;  // pages past the context: the box is out of bounds and reads zeros
        if (blk < nblk) {
          id = __ldg(table + blk);
          if (id < 0 || id >= p.num_blocks) atomicOr(&g_prefill_error, kErrBadBlockId);
        }
        const uint32_t dst = sbase + L::kStageOff + st * L::kStageBytes + kv * L::kTileBytes +
                             h * L::kHalf + b * 2048;
        tma_load_4d(dst, kv ? &tmap_v : &tmap_k, bars + 8 * (kKvFull0 + st), h * 64, kvh, 0, id);
      }
      if (lane == 0) issued[st] = j / kPfStages + 1;
    }
    // Drain: wait (bounded, regardless of aborts) for every phase issued, so no
    // copy lands in shared memory after the CTA exits.
    if (lane == 0 && *abort_flag) {
      if (issued_q) (void)mbar_wait_bounded(bars + 8 * kQFull, 0);
      for (int s = 0; s < kPfStages; ++s)
        if (issued[s] > 0) (void)mbar_wait_bounded(bars + 8 * (kKvFull0 + s), (issued[s] - 1) & 1);
    }
  }
  else if (warp == kPfMmaWarp) {
    // ================= MMA issuer (one thread) =================
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(128, kPfKvTile, 0, 0);
      constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, 0, 1);
      bool ok = pf_wait(bars + 8 * kQFull, 0, abort_flag);
      // S_j = Q K_j^T into TMEM columns [128 (j % 2), +128)
      auto issue_s = [&](int j) -> bool {
        const int st = j % kPfStages;
        if (!pf_wait(bars + 8 * (kKvFull0 + st), (j / kPfStages) & 1, abort_flag)) return false;
        tc_fence_after();
        const uint32_t k_smem = sbase + L::kStageOff + st * L::kStageBytes;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * L::kHalf + (k & 3) * 32;
          umma_bf16(tmem + (j & 1) * 128, smem_desc_sw128(q_smem + off, 16, 1024),
                    smem_desc_sw128(k_smem + off, 16, 1024), kIdescS, k > 0);
        }
        umma_commit(bars + 8 * (kSFull0 + (j & 1)));
        return true;
      };
      for (int j = 0; ok && j < ntiles && j < 2; ++j) ok = issue_s(j);
      for (int j = 0; ok && j < ntiles; ++j) {
        if (!pf_wait(bars + 8 * kPFull, j & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // O += P_j V_j: P K-major (rows x keys), V MN-major (keys x d) from the pool layout
        const uint32_t v_smem = sbase + L::kStageOff + (j % kPfStages) * L::kStageBytes +
                                L::kTileBytes;
#pragma unroll
        for (int k = 0; k < kPfKvTile / 16; ++k) {
          const uint32_t poff = (k >> 2) * L::kHalf + (k & 3) * 32;
          const uint64_t vdesc = smem_desc_sw128(v_smem + k * 2048, L::kHalf, 1024);
          umma_bf16(tmem + 256, smem_desc_sw128(p_smem + poff, 16, 1024), vdesc, kIdescPV,
                    (j > 0 || k > 0) ? 1u : 0u);
          umma_bf16(tmem + 256, smem_desc_sw128(p_smem + L::kPBytes + poff, 16, 1024), vdesc,
                    kIdescPV, 1u);
        }
        umma_commit(bars + 8 * (kKvEmpty0 + (j % kPfStages)));
        umma_commit(bars + 8 * kODone);
        if (j + 2 < ntiles) ok = issue_s(j + 2);
      }
      if (!ok) pf_abort(abort_flag);
      // every MMA issued has completed before tensor memory is released
      umma_commit(bars + 8 * kDrain);
      (void)mbar_wait_bounded(bars + 8 * kDrain, 0);
    }
    __syncwarp();
  } else {
    // ================= softmax / correction / epilogue (warps 0-3) =================
    const int r = warp * 32 + lane;  // row = TMEM lane
    const int token = r / G, head = r - (r / G) * G;
    const int tok = t0 + token;
    const bool valid_row = tok < n;
    // rows past the chunk compute finite garbage over the whole context and are not stored
    const int limit = (p.causal && valid_row) ? (ctx - n + tok) : (ctx - 1);
    const uint32_t lane_base = tmem + (uint32_t(warp * 32) << 16);
    float m_used = -INFINITY, lsum = 0.f;
    bool ok = true;
    int j = 0;
    for (; j < ntiles; ++j) {
      ok = __all_sync(0xffffffffu, pf_wait(bars + 8 * (kSFull0 + (j & 1)), (j >> 1) & 1,
                                           abort_flag));
      if (!ok) break;
      tc_fence_after();
      float s[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + (j & 1) * 128 + c * 32, s[c]);
      tmem_wait_ld();
      const int key0 = j * kPfKvTile;
      const bool need_mask = key0 + kPfKvTile - 1 > limit;
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float x = s[c][i] * p.scale_log2;
          if (need_mask && key0 + c * 32 + i > limit) x = -INFINITY;
          s[c][i] = x;
          mx = fmaxf(mx, x);
        }
      if (j > 0) {
        // PV_{j-1} done: the P buffer is free and O is stable
        ok = __all_sync(0xffffffffu, pf_wait(bars + 8 * kODone, (j - 1) & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
      }
      const bool resc = mx > m_used + kRescaleThreshold;
      if (__any_sync(0xffffffffu, resc)) {
        const float m_new = resc ? mx : m_used;
        const float alpha = ex2(m_used - m_new);  // 0 when m_used is -inf, 1 when unchanged
        if (j > 0) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tmem_ld32(lane_base + 256 + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(lane_base + 256 + c * 32, o);
          }
          tmem_wait_st();
        }
        lsum *= alpha;
        m_used = m_new;
      }
      // P = 2^(x - m_used) as bf16 into the K-major swizzled P tile
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int g8 = 0; g8 < 4; ++g8) {
          float e[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            e[u] = ex2(s[c][g8 * 8 + u] - m_used);
            lsum += e[u];
          }
          const int key = c * 32 + g8 * 8;  // first of 8 keys in this 16-byte chunk
          const int half = key >> 6, chunk = (key & 63) >> 3;
          const uint32_t addr = p_smem + half * L::kHalf + r * 128 + ((chunk ^ (r & 7)) << 4);
          uint32_t w[4], wl[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            w[u] = pack_bf16x2(e[2 * u], e[2 * u + 1]);
            wl[u] = pack_bf16x2(e[2 * u] - bf16_lo_to_f32(w[u]),
                                e[2 * u + 1] - bf16_hi_to_f32(w[u]));
          }
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]),
                       "r"(w[1]), "r"(w[2]), "r"(w[3])
                       : "memory");
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr + L::kPBytes),
                       "r"(wl[0]), "r"(wl[1]), "r"(wl[2]), "r"(wl[3])
                       : "memory");
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + 8 * kPFull);
    }
    if (!ok) {
      if (lane == 0) pf_abort(abort_flag);
    } else {
      // epilogue: wait for the last PV, then out = O / l
      ok = __all_sync(0xffffffffu,
                      pf_wait(bars + 8 * kODone, (ntiles - 1) & 1, abort_flag));
      if (!ok) {
        if (lane == 0) pf_abort(abort_flag);
      } else {
        tc_fence_after();
        const float inv = 1.f / lsum;
        float* orow = p.out + (size_t(qs + tok) * p.q_heads + size_t(kvh) * G + head) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32(lane_base + 256 + c * 32, o);
          tmem_wait_ld();
          if (valid_row) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4*>(orow + c * 32 + i) =
                  make_float4(o[i] * inv, o[i + 1] * inv, o[i + 2] * inv, o[i + 3] * inv);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kPfTmemCols);
  }
}

template <int D, int G>
static cudaError_t launch_prefill_t(const PrefillParams& prm, const CUtensorMap* tq,
                                    const CUtensorMap* tk, const CUtensorMap* tv,
                                    cudaStream_t stream) {
  using L = PrefillSmem<D>;
  constexpr int TPT = kPfRows / G;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(paged_prefill_kernel<D, G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid((prm.max_q_len + TPT - 1) / TPT, prm.num_seqs * prm.kv_heads);
  paged_prefill_kernel<D, G><<<grid, kPfThreads, L::kSmemBytes, stream>>>(*tq, *tk, *tv, prm);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_prefill_d(const PrefillParams& prm, int group, const CUtensorMap* tq,
                                    const CUtensorMap* tk, const CUtensorMap* tv,
                                    cudaStream_t st) {
  switch (group) {
    case 1: return launch_prefill_t<D, 1>(prm, tq, tk, tv, st);
    case 2: return launch_prefill_t<D, 2>(prm, tq, tk, tv, st);
    case 4: return launch_prefill_t<D, 4>(prm, tq, tk, tv, st);
    case 8: return launch_prefill_t<D, 8>(prm, tq, tk, tv, st);
    case 16: return launch_prefill_t<D, 16>(prm, tq, tk, tv, st);
    default: return cudaErrorInvalidValue;
  }
}

int prefill_rows_per_tile() { return kPfRows; }

cudaError_t launch_paged_prefill(const PrefillArgs& a, const CUtensorMap* tmap_q,
                                 const CUtensorMap* tmap_k, const CUtensorMap* tmap_v,
                                 cudaStream_t stream) {
  PrefillParams prm;
  prm.q_start = a.q_start;
  prm.block_tables = a.block_tables;
  prm.context_lens = a.context_lens;
  prm.out = a.out;
  prm.num_seqs = a.num_seqs;
  prm.q_heads = a.q_heads;
  prm.kv_heads = a.kv_heads;
  prm.num_blocks = a.num_blocks;
  prm.max_blocks_per_seq = a.max_blocks_per_seq;
  prm.total_q = a.total_q;
  prm.max_q_len = a.max_q_len;
  prm.causal = a.causal;
  prm.scale_log2 = a.scale_log2;
  const int group = a.q_heads / a.kv_heads;
  if (a.d_head == 128) return launch_prefill_d<128>(prm, group, tmap_q, tmap_k, tmap_v, stream);
  if (a.d_head == 64) return launch_prefill_d<64>(prm, group, tmap_q, tmap_k, tmap_v, stream);
  return cudaErrorInvalidValue;
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
