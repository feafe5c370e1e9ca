// The tensor-core chunked-prefill item (two 128-row query tiles of one
// sequence x KV head, computed by a whole CTA of kPfThreads threads) shared
// by the prefill kernels and the fused mixed-step kernel, with its shared
// memory layout, barrier roles and dispatch order.  Each translation unit
// that includes this header gets its own device error word g_prefill_error.
#pragma once

#include <algorithm>
#include <climits>
#include <type_traits>

#include "pkv_device.cuh"
#include "pkv_tcgen05.cuh"

namespace pkv {

static __device__ unsigned g_prefill_error = 0;

constexpr int kPfRows = 128;          // query rows per Q tile (tokens x heads)
constexpr int kPfQTiles = 2;          // Q tiles per CTA, one softmax warpgroup each
constexpr int kPfKvTile = 128;        // keys per K/V tile (8 pages of 16)
constexpr int kPfKStages = 3;         // K tile ring (freed once both S products are done)
constexpr int kPfVStages = 2;         // V tile ring (freed once both PV products are done)
constexpr int kPfThreads = 352;       // 2 softmax warpgroups + K/Q TMA + MMA + V TMA warps
constexpr int kPfProducerWarp = 8;    // loads Q and K
constexpr int kPfMmaWarp = 9;
constexpr int kPfVProducerWarp = 10;  // loads V
constexpr uint32_t kPfTmemCols = 512; // per Q tile t: S_t / P_t at 256 t, O_t at 256 t + 128
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows by > x256

template <int D>
struct PrefillSmem {
  static constexpr int kHalf = kPfRows * 128;                // 128 rows x 64 bf16 (16 KB)
  static constexpr int kQTileBytes = (D / 64) * kHalf;
  static constexpr int kTileBytes = (D / 64) * kHalf;        // K or V: 128 keys x D
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kPfQTiles * kQTileBytes;
  static constexpr int kVOff = kKOff + kPfKStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kPfVStages * kTileBytes;
  // q_full, k_full[3], k_empty[3], v_full[2], v_empty[2], s_full[2], p_full[2], o_done[2], drain
  static constexpr int kNumBars = 18;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;     // tmem base, abort flag
  static constexpr int kUsed = kMiscOff + 16 + 1024;          // + alignment slack
  // One CTA per SM: it holds all 512 TMEM columns.
  static constexpr int kSmemBytes = kUsed > 120 * 1024 ? kUsed : 120 * 1024;
  static_assert(kSmemBytes <= 232448, "prefill tile does not fit in shared memory");
};

enum PfBar { kQFull = 0, kKFull0 = 1, kKEmpty0 = 4, kVFull0 = 7, kVEmpty0 = 9, kSFull0 = 11,
             kPFull0 = 13, kODone0 = 15, kDrain = 17 };

struct PrefillParams {
  const int32_t* q_start;       // null: one sequence owning all total_q rows
  const int32_t* block_tables;
  const int32_t* context_lens;  // null: the context length is `context_len`
  float* out;
  float* lse;                   // optional [total_q][q_heads] log2-sum-exp of each row
  int num_seqs, q_heads, kv_heads, num_blocks, max_blocks_per_seq, total_q, max_q_len;
  int causal;
  int context_len;
  float scale_log2;
  float out_scale;              // multiplies the output (1, or v_scale over FP8 pools)
  const int32_t* v_block_tables;  // null: V pages use block_tables
  int v_num_blocks;             // blocks of the V pool
  // persistent mode: CTAs take items (pair, query tile) from this counter,
  // zero on entry, in the grid mode's order (item_pair_tile); null: one
  // item per CTA from the grid
  int* work_counter;
  int num_items;                // pairs * tiles_per_pair
  int tiles_per_pair;           // CTA-sized query tiles of the longest chunk
  int out_bf16;                 // nonzero: out holds bf16, rounded to nearest even
  const int32_t* seq_order;     // [num_seqs] dispatch order of the sequences, or null
  // [num_seqs] row of block_tables each sequence's pages are in (null: its
  // own row): a prefix group's queries read the group leader's row
  const int32_t* table_rows = nullptr;
  int allow_empty = 0;          // nonzero: a context of 0 is skipped without a flag
  int defer_wait = 0;           // nonzero: wait for the previous grid at the end, not the start
  // nonzero: float32 rows of whole warps leave through the output tensor map
  // (tmap_o: d_head x q_heads x total_q, box 32 columns x G heads x 32/G
  // tokens, 128-byte swizzled), staged in the then idle K/V rings
  int o_tma = 0;
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

// One item: the two query tiles `cta_tile` of pair (sequence x KV head)
// `pair`, computed by the whole CTA.  Barriers are set up at the start; at
// the end every copy, MMA and tensor-memory access of the item has completed
// and the CTA has synchronised, so the next item can reuse everything.
// F16PV: V is an f16 pool and P enters the PV product as one f16 operand;
// otherwise V is bf16 and P enters as bf16 hi + lo.
template <int D, int G, bool F16PV>
__device__ __forceinline__ void prefill_item(const CUtensorMap& tmap_q, const CUtensorMap& tmap_k,
                                             const CUtensorMap& tmap_v, const CUtensorMap& tmap_o,
                                             const PrefillParams& p, uint8_t* smem, uint32_t tmem,
                                             int pair, int cta_tile) {
  using L = PrefillSmem<D>;
  constexpr int TPT = kPfRows / G;          // query tokens per Q tile
  constexpr int TPC = kPfQTiles * TPT;      // query tokens per CTA
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + L::kBarOff;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seq = pair / p.kv_heads;
  const int kvh = pair - seq * p.kv_heads;

  // ---- per-item bounds (uniform over the CTA, so early exits are safe)
  const int qs = p.q_start ? __ldg(p.q_start + seq) : 0;
  const int qe = p.q_start ? __ldg(p.q_start + seq + 1) : p.total_q;
  const int ctx = p.context_lens ? __ldg(p.context_lens + seq) : p.context_len;
  const int n = qe - qs;
  const bool bad_range = qs < 0 || n < 0 || qe > p.total_q;
  if (!bad_range && n == 0) return;  // nothing to compute for this sequence
  if (!bad_range && ctx == 0 && p.allow_empty) return;  // an empty prefix group
  // A chunk longer than max_q_len would have tiles the launch does not cover:
  // the whole sequence is rejected rather than computed in part.
  if (bad_range || (p.causal && n > ctx) || ctx <= 0 || ctx > p.max_blocks_per_seq * 16 ||
      n > p.max_q_len) {
    if (cta_tile == 0 && threadIdx.x == 0) atomicOr(&g_prefill_error, kErrBadQueryRange);
    return;
  }
  const int t0 = cta_tile * TPC;
  if (t0 >= n) return;
  const int tok_valid = min(TPC, n - t0);
  const int kv_end = p.causal ? (ctx - n + t0 + tok_valid) : ctx;  // keys [0, kv_end)
  const int ntiles = (kv_end + kPfKvTile - 1) / kPfKvTile;
  const int nblk = (ctx + 15) / 16;

  // ---- set-up: barriers (producer lane 0)
  if (warp == kPfProducerWarp && lane == 0) {
    mbar_init(bars + 8 * kQFull, 1);
    for (int s = 0; s < kPfKStages; ++s) {
      mbar_init(bars + 8 * (kKFull0 + s), 1);
      mbar_init(bars + 8 * (kKEmpty0 + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bars + 8 * (kVFull0 + s), 1);
      mbar_init(bars + 8 * (kVEmpty0 + s), 1);
      mbar_init(bars + 8 * (kSFull0 + s), 1);
      mbar_init(bars + 8 * (kPFull0 + s), 4);
      mbar_init(bars + 8 * (kODone0 + s), 1);
    }
    mbar_init(bars + 8 * kDrain, 1);
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == kPfProducerWarp || warp == kPfVProducerWarp) {
    // ============ TMA producers: warp 8 loads Q and the K ring, warp 10 the V ring ============
    const bool is_v = warp == kPfVProducerWarp;
    const int stages = is_v ? kPfVStages : kPfKStages;
    const uint32_t ring = sbase + (is_v ? L::kVOff : L::kKOff);
    const uint32_t full0 = bars + 8 * (is_v ? kVFull0 : kKFull0);
    const uint32_t empty0 = bars + 8 * (is_v ? kVEmpty0 : kKEmpty0);
    const CUtensorMap* map = is_v ? &tmap_v : &tmap_k;
    int issued_q = 0, issued[kPfKStages] = {0, 0, 0};
    if (!is_v && lane == 0) {
      tma_prefetch_desc(&tmap_q);
      tma_prefetch_desc(&tmap_k);
      mbar_arrive_expect_tx(bars + 8 * kQFull, kPfQTiles * L::kQTileBytes);
#pragma unroll
      for (int t = 0; t < kPfQTiles; ++t)
#pragma unroll
        for (int h = 0; h < D / 64; ++h)
          tma_load_3d(sbase + L::kQOff + t * L::kQTileBytes + h * L::kHalf, &tmap_q,
                      bars + 8 * kQFull, h * 64, kvh * G, qs + t0 + t * TPT);
      issued_q = 1;
    }
    if (is_v && lane == 0) tma_prefetch_desc(&tmap_v);
    const bool own_table = is_v && p.v_block_tables;  // a scratch pool's table: one row per sequence
    const int row = (!own_table && p.table_rows) ? __ldg(p.table_rows + seq) : seq;
    const int32_t* table = (own_table ? p.v_block_tables : p.block_tables) +
                           size_t(row) * p.max_blocks_per_seq;
    const int pool_blocks = is_v ? p.v_num_blocks : p.num_blocks;
    constexpr int kLoads = 8 * (D / 64);  // 8 pages x D/64 column halves
    for (int j = 0; j < ntiles; ++j) {
      const int st = j % stages;
      if (j >= stages) {
        const bool ok = __all_sync(0xffffffffu,
                                   pf_wait(empty0 + 8 * st, ((j / stages) - 1) & 1, abort_flag));
        if (!ok) {
          if (lane == 0) pf_abort(abort_flag);
          break;
        }
      }
      if (lane == 0) mbar_arrive_expect_tx(full0 + 8 * st, L::kTileBytes);
      __syncwarp();
      if (lane < kLoads) {
        const int b = lane / (D / 64);
        const int h = lane % (D / 64);
        const int blk = j * 8 + b;
        int id = -1;  // pages past the context: the box is out of bounds and reads zeros
        if (blk < nblk) {
          id = __ldg(table + blk);
          if (id < 0 || id >= pool_blocks) atomicOr(&g_prefill_error, kErrBadBlockId);
        }
        tma_load_4d(ring + st * L::kTileBytes + h * L::kHalf + b * 2048, map, full0 + 8 * st,
                    h * 64, kvh, 0, id);
      }
      if (lane == 0) issued[st] = j / stages + 1;
    }
    // Drain: wait (bounded, regardless of aborts) for every phase issued, so no
    // copy lands in shared memory after the CTA exits.
    if (lane == 0 && *abort_flag) {
      if (issued_q) (void)mbar_wait_bounded(bars + 8 * kQFull, 0);
      for (int s = 0; s < stages; ++s)
        if (issued[s] > 0) (void)mbar_wait_bounded(full0 + 8 * s, (issued[s] - 1) & 1);
    }
  }
  else if (warp == kPfMmaWarp) {
    // ================= MMA issuer (one thread) =================
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(128, kPfKvTile, 0, 0);
      constexpr uint32_t kIdescPV =
          F16PV ? idesc_f16_f32(128, D, 0, 1) : idesc_bf16_f32(128, D, 0, 1);
      // S_t(j) = Q_t K_j^T into TMEM columns [256 t, 256 t + 128)
      auto issue_s = [&](int t, int j) {
        const uint32_t q_smem = sbase + L::kQOff + t * L::kQTileBytes;
        const uint32_t k_smem = sbase + L::kKOff + (j % kPfKStages) * L::kTileBytes;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * L::kHalf + (k & 3) * 32;
          umma_bf16(tmem + t * 256, smem_desc_sw128(q_smem + off, 16, 1024),
                    smem_desc_sw128(k_smem + off, 16, 1024), kIdescS, k > 0);
        }
        umma_commit(bars + 8 * (kSFull0 + t));
      };
      // O_t += P_t(j) V_j: P (bf16 hi, lo -- or one f16) read from TMEM over S_t's
      // columns, V the MN-major operand (keys x d) straight from the pool layout
      auto issue_pv = [&](int t, int j) {
        const uint32_t v_smem = sbase + L::kVOff + (j % kPfVStages) * L::kTileBytes;
#pragma unroll
        for (int k = 0; k < kPfKvTile / 16; ++k) {
          const uint64_t vdesc = smem_desc_sw128(v_smem + k * 2048, L::kHalf, 1024);
          // keys [16 k, 16 k + 16): hi in column 64 (k / 4) + 8 (k % 4), lo 32 columns on
          const uint32_t a_hi = tmem + t * 256 + 64 * (k >> 2) + 8 * (k & 3);
          umma_bf16_ts(tmem + t * 256 + 128, a_hi, vdesc, kIdescPV, (j > 0 || k > 0) ? 1u : 0u);
          if constexpr (!F16PV) umma_bf16_ts(tmem + t * 256 + 128, a_hi + 32, vdesc, kIdescPV, 1u);
        }
        umma_commit(bars + 8 * (kODone0 + t));
      };
      // Rows of the context's last page past its length may hold anything,
      // NaN included.  Their P is 0; zeroing their V rows in shared memory
      // (whole 128-byte rows, so the swizzle does not matter) keeps 0 * V
      // exactly 0.  Generic stores, then a proxy fence for the tensor core.
      const int tail_rows = ctx & 15;
      const int j_tail = (nblk - 1) / 8;
      auto clear_tail = [&](int j) {
        const uint32_t page = sbase + L::kVOff + (j % kPfVStages) * L::kTileBytes +
                              ((nblk - 1) % 8) * 2048;
        for (int h = 0; h < D / 64; ++h)
          for (int r = tail_rows; r < 16; ++r)
#pragma unroll
            for (int c = 0; c < 8; ++c) st_shared_zero16(page + h * L::kHalf + r * 128 + c * 16);
        fence_proxy_async_smem();
      };
      auto ready = [&](uint32_t full0, int stages, int j) {
        const bool r = pf_wait(full0 + 8 * (j % stages), (j / stages) & 1, abort_flag);
        if (r) tc_fence_after();
        return r;
      };
      const uint32_t kfull0 = bars + 8 * kKFull0, vfull0 = bars + 8 * kVFull0;
      bool ok = pf_wait(bars + 8 * kQFull, 0, abort_flag) && ready(kfull0, kPfKStages, 0);
      if (ok) {
        issue_s(0, 0);
        issue_s(1, 0);
        umma_commit(bars + 8 * kKEmpty0);  // K_0 free once both S products are done
      }
      // Ping-pong: the tensor core works on one Q tile while the other's softmax runs.
      for (int j = 0; ok && j < ntiles; ++j) {
        if (!pf_wait(bars + 8 * kPFull0, j & 1, abort_flag) || !ready(vfull0, kPfVStages, j)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (tail_rows && j == j_tail) clear_tail(j);
        issue_pv(0, j);
        const bool more = j + 1 < ntiles;
        if (more) {
          if (!ready(kfull0, kPfKStages, j + 1)) {
            ok = false;
            break;
          }
          issue_s(0, j + 1);
        }
        if (!pf_wait(bars + 8 * (kPFull0 + 1), j & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_pv(1, j);
        umma_commit(bars + 8 * (kVEmpty0 + j % kPfVStages));  // V_j free after both PV
        if (more) {
          issue_s(1, j + 1);
          umma_commit(bars + 8 * (kKEmpty0 + (j + 1) % kPfKStages));  // K_{j+1} free
        }
      }
      if (!ok) pf_abort(abort_flag);
      // every MMA issued has completed before tensor memory is released
      umma_commit(bars + 8 * kDrain);
      (void)mbar_wait_bounded(bars + 8 * kDrain, 0);
      if (ok) {
        // ... and every commit has arrived before the barriers are set up
        // again for the next item: the last phase of each ring slot's
        // empty barrier (tile j was committed to slot j % stages)
        for (int s = 0; s < kPfKStages && s < ntiles; ++s) {
          const int last = s + (ntiles - 1 - s) / kPfKStages * kPfKStages;
          (void)mbar_wait_bounded(bars + 8 * (kKEmpty0 + s), (last / kPfKStages) & 1);
        }
        for (int s = 0; s < kPfVStages && s < ntiles; ++s) {
          const int last = s + (ntiles - 1 - s) / kPfVStages * kPfVStages;
          (void)mbar_wait_bounded(bars + 8 * (kVEmpty0 + s), (last / kPfVStages) & 1);
        }
      }
    }
    __syncwarp();
  } else {
    // ============ softmax / correction / epilogue: warpgroup wg owns Q tile wg ============
    const int wg = warp >> 2;
    const int r = (warp & 3) * 32 + lane;  // row of the Q tile = TMEM lane
    const int token = r / G, head = r - (r / G) * G;
    const int tok = t0 + wg * TPT + token;
    const bool valid_row = tok < n;
    // rows past the chunk compute finite garbage over the whole context and are not stored
    const int limit = (p.causal && valid_row) ? (ctx - n + tok) : (ctx - 1);
    const uint32_t lane_base = tmem + (uint32_t((warp & 3) * 32) << 16);
    const uint32_t s_col = wg * 256, o_col = wg * 256 + 128;
    const uint32_t s_full = bars + 8 * (kSFull0 + wg), p_full = bars + 8 * (kPFull0 + wg);
    const uint32_t o_done = bars + 8 * (kODone0 + wg);
    float m_used = -INFINITY, lsum = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      ok = __all_sync(0xffffffffu, pf_wait(s_full, j & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      const int key0 = j * kPfKvTile;
      const bool need_mask = key0 + kPfKvTile - 1 > limit;
      if constexpr (F16PV) {
        // P of keys [64 g, 64 g + 64) as packed f16 pairs, held in registers
        // until the tile is settled and then stored over S's columns
        uint32_t pk[64];
        float tsum;
        const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
        // No max pass while the running max may stay, on masked tiles too
        // (the exponentials apply each row's mask).  The first tile seeds
        // the running max from its first 32 keys and keeps it when the sum
        // of the rounded weights allows, as any other tile does.
        bool fast = __all_sync(0xffffffffu, j > 0);
        bool seeded = false;
        for (;;) {
          if (!fast && j == 0 && !seeded) {
            // key 0 is visible to every row, so the seed is finite
            float va[32];
            tmem_ld32(lane_base + s_col, va);
            tmem_wait_ld();
            const bool neg = p.scale_log2 < 0.f;  // uniform over the CTA
            float ex[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float a = neg ? -va[i] : va[i];
              if (i <= limit) ex[i & 3] = fmaxf(ex[i & 3], a);
            }
            m_used = fmaxf(fmaxf(ex[0], ex[1]), fmaxf(ex[2], ex[3])) * fabsf(p.scale_log2);
            seeded = true;
            fast = true;
          } else if (!fast) {
            float ex[8];
#pragma unroll
            for (int a = 0; a < 8; ++a) ex[a] = -INFINITY;
            const bool neg = p.scale_log2 < 0.f;  // uniform over the CTA
#pragma unroll
            for (int c = 0; c < 4; c += 2) {
              float va[32], vb[32];
              tmem_ld32(lane_base + s_col + c * 32, va);
              tmem_ld32(lane_base + s_col + c * 32 + 32, vb);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const float a = neg ? -va[i] : va[i], b = neg ? -vb[i] : vb[i];
                if (key0 + c * 32 + i <= limit) ex[i & 7] = fmaxf(ex[i & 7], a);
                if (key0 + c * 32 + 32 + i <= limit) ex[i & 7] = fmaxf(ex[i & 7], b);
              }
            }
            const float ext = fmaxf(fmaxf(fmaxf(ex[0], ex[1]), fmaxf(ex[2], ex[3])),
                                    fmaxf(fmaxf(ex[4], ex[5]), fmaxf(ex[6], ex[7])));
            const float mx = ext == -INFINITY ? -INFINITY : ext * fabsf(p.scale_log2);
            const bool resc = mx > m_used + kRescaleThreshold;
            if (__any_sync(0xffffffffu, resc)) {
              const float m_new = resc ? mx : m_used;
              const float alpha = ex2(m_used - m_new);  // 0 when m_used is -inf, 1 when unchanged
              if (j > 0) {
                // PV_{j-1} must be done before O is rescaled
                ok = __all_sync(0xffffffffu, pf_wait(o_done, (j - 1) & 1, abort_flag));
                if (!ok) break;
                tc_fence_after();
                const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
                for (int c = 0; c < D / 16; ++c) {
                  float o[16];
                  tmem_ld16(lane_base + o_col + c * 16, o);
                  tmem_wait_ld();
#pragma unroll
                  for (int i = 0; i < 16; i += 2)
                    f2_unpack(f2_mul(f2_pack(o[i], o[i + 1]), a2), o[i], o[i + 1]);
                  tmem_st16(lane_base + o_col + c * 16, o);
                }
              }
              lsum *= alpha;
              m_used = m_new;
            }
          }
          // P = 2^(x - m_used) for all keys, and the sum of the rounded weights
          const uint64_t nm2 = f2_pack(-m_used, -m_used);
          float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            float va[32], vb[32];
            tmem_ld32(lane_base + s_col + 64 * g, va);
            tmem_ld32(lane_base + s_col + 64 * g + 32, vb);
            tmem_wait_ld();
            if (!need_mask) {
#pragma unroll
              for (int u = 0; u < 32; ++u) {
                const int kk = 2 * u;
                const float s0 = kk < 32 ? va[kk] : vb[kk - 32];
                const float s1 = kk < 32 ? va[kk + 1] : vb[kk - 31];
                float x0, x1;
                f2_unpack(f2_fma(f2_pack(s0, s1), sc2, nm2), x0, x1);
                pk[32 * g + u] = pack_f16x2_rn(ex2(x0), ex2(x1));
                ls[u & 3] = add_f16x2_to_f32(pk[32 * g + u], ls[u & 3]);
              }
            } else {
#pragma unroll
              for (int u = 0; u < 32; ++u) {
                const int kk = 2 * u;
                const float s0 = kk < 32 ? va[kk] : vb[kk - 32];
                const float s1 = kk < 32 ? va[kk + 1] : vb[kk - 31];
                const int key = key0 + 64 * g + kk;
                float x0, x1;
                f2_unpack(f2_fma(f2_pack(s0, s1), sc2, nm2), x0, x1);
                pk[32 * g + u] = pack_f16x2_rn(key <= limit ? ex2(x0) : 0.f,
                                               key + 1 <= limit ? ex2(x1) : 0.f);
                ls[u & 3] = add_f16x2_to_f32(pk[32 * g + u], ls[u & 3]);
              }
            }
          }
          tsum = (ls[0] + ls[1]) + (ls[2] + ls[3]);
          // every weight <= tsum; NaN or inf fail the test and take the max pass
          if (!fast || __all_sync(0xffffffffu, tsum <= 256.f)) break;
          fast = false;
        }
        if (!ok) break;
        lsum += tsum;
        tmem_st32u(lane_base + s_col, *reinterpret_cast<const uint32_t(*)[32]>(pk));
        tmem_st32u(lane_base + s_col + 64, *reinterpret_cast<const uint32_t(*)[32]>(pk + 32));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
        continue;
      }
      // hi + lo P keeps fp32's exponent range, so a stale running max only
      // has to keep the exponentials finite.  The max pass is skipped: the
      // first tile seeds the running max from its first 32 keys (key 0 is
      // visible to every row), and the exponentials are taken against m_used,
      // 64 keys at a time with each row's causal mask, a group kept while
      // every row's sum over it stays <= 2^64 (every weight is at most that
      // sum).  A first group that fails leaves S intact for the two-pass path
      // below; a second group that fails after the first was stored raises
      // the max from its own visible scores and rescales O, the row sum and
      // the stored first group (hi + lo is exact in fp32) before recomputing.
      if (j == 0 && p.scale_log2 > 0.f) {
        float va[32];
        tmem_ld32(lane_base + s_col, va);
        tmem_wait_ld();
        float ex[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (i <= limit) ex[i & 3] = fmaxf(ex[i & 3], va[i]);
        m_used = fmaxf(fmaxf(ex[0], ex[1]), fmaxf(ex[2], ex[3])) * p.scale_log2;
      }
      if (p.scale_log2 > 0.f) {  // uniform over the CTA
        const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
        bool two_pass = false;
        for (int g = 0; g < 2; ++g) {
          float va[32], vb[32];
          tmem_ld32(lane_base + s_col + 64 * g, va);
          tmem_ld32(lane_base + s_col + 64 * g + 32, vb);
          tmem_wait_ld();
          for (int attempt = 0;; ++attempt) {
            uint32_t hi[32], lo[32];
            const uint64_t nm2 = f2_pack(-m_used, -m_used);
            uint64_t ls2[2] = {0ull, 0ull};
            // arithmetic only: rows differ in need_mask
            auto exps = [&](auto masked) {
#pragma unroll
              for (int u = 0; u < 32; ++u) {
                const int kk = 2 * u;
                const float s0 = kk < 32 ? va[kk] : vb[kk - 32];
                const float s1 = kk < 32 ? va[kk + 1] : vb[kk - 31];
                float x0, x1;
                f2_unpack(f2_fma(f2_pack(s0, s1), sc2, nm2), x0, x1);
                float e0 = ex2(x0), e1 = ex2(x1);
                if constexpr (decltype(masked)::value) {
                  const int key = key0 + 64 * g + kk;
                  e0 = key <= limit ? e0 : 0.f;
                  e1 = key + 1 <= limit ? e1 : 0.f;
                }
                const uint64_t e = f2_pack(e0, e1);
                ls2[u & 1] = f2_add(ls2[u & 1], e);
                hi[u] = pack_bf16x2(e0, e1);
                float r0, r1;
                f2_unpack(f2_sub(e, f2_pack(bf16_lo_to_f32(hi[u]), bf16_hi_to_f32(hi[u]))), r0,
                          r1);
                lo[u] = pack_bf16x2(r0, r1);
              }
            };
            if (need_mask) exps(std::true_type{});
            else exps(std::false_type{});
            float a0, a1, b0, b1;
            f2_unpack(ls2[0], a0, a1);
            f2_unpack(ls2[1], b0, b1);
            const float gsum = (a0 + a1) + (b0 + b1);
            // NaN or inf fail the test
            if (attempt > 0 || __all_sync(0xffffffffu, gsum <= 18446744073709551616.f)) {
              lsum += gsum;
              tmem_st32u(lane_base + s_col + 64 * g, hi);
              tmem_st32u(lane_base + s_col + 64 * g + 32, lo);
              break;
            }
            if (g == 0) {  // nothing stored yet
              two_pass = true;
              break;
            }
            // the max rose within the second group: take it from its visible scores
            float ex[8];
#pragma unroll
            for (int a = 0; a < 8; ++a) ex[a] = -INFINITY;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int key = key0 + 64 * g + i;
              ex[i & 7] = max3f(ex[i & 7], key <= limit ? va[i] : -INFINITY,
                                key + 32 <= limit ? vb[i] : -INFINITY);
            }
            const float ext = fmaxf(fmaxf(fmaxf(ex[0], ex[1]), fmaxf(ex[2], ex[3])),
                                    fmaxf(fmaxf(ex[4], ex[5]), fmaxf(ex[6], ex[7])));
            const float m_new = fmaxf(m_used, ext * p.scale_log2);
            const float alpha = ex2(m_used - m_new);
            const uint64_t a2 = f2_pack(alpha, alpha);
            // PV_{j-1} must be done before O is rescaled
            ok = __all_sync(0xffffffffu, pf_wait(o_done, (j - 1) & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              float o[32];
              tmem_ld32(lane_base + o_col + c * 32, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; i += 2)
                f2_unpack(f2_mul(f2_pack(o[i], o[i + 1]), a2), o[i], o[i + 1]);
              tmem_st32(lane_base + o_col + c * 32, o);
            }
            // the first group's stored P: hi + lo (exact in fp32) times alpha,
            // split again, 16 columns (32 keys) at a time
            tmem_wait_st();
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
              float ph[16], pl[16];
              tmem_ld16(lane_base + s_col + 16 * c, ph);
              tmem_ld16(lane_base + s_col + 32 + 16 * c, pl);
              tmem_wait_ld();
#pragma unroll
              for (int u = 0; u < 16; ++u) {
                const uint32_t hw = __float_as_uint(ph[u]), lw = __float_as_uint(pl[u]);
                float e0, e1;
                f2_unpack(f2_mul(f2_add(f2_pack(bf16_lo_to_f32(hw), bf16_hi_to_f32(hw)),
                                        f2_pack(bf16_lo_to_f32(lw), bf16_hi_to_f32(lw))),
                                 a2),
                          e0, e1);
                const uint32_t h = pack_bf16x2(e0, e1);
                ph[u] = __uint_as_float(h);
                pl[u] = __uint_as_float(pack_bf16x2(e0 - bf16_lo_to_f32(h), e1 - bf16_hi_to_f32(h)));
              }
              tmem_st16(lane_base + s_col + 16 * c, ph);
              tmem_st16(lane_base + s_col + 32 + 16 * c, pl);
            }
            lsum *= alpha;
            m_used = m_new;
          }
          if (!ok || two_pass) break;
        }
        if (!ok) break;
        if (!two_pass) {
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(p_full);
          continue;
        }
      }
      // pass 1: row max.  On unmasked tiles the max is taken over the raw
      // scores and scaled once (scale > 0 keeps the order; scale < 0 flips it).
      float mx;
      {
        float va[32], vb[32];
        // the extreme that becomes the max after scaling: max for scale >= 0,
        // min (taken as the max of the negated scores) for scale < 0
        const bool neg = p.scale_log2 < 0.f;  // uniform over the CTA
        // 8 independent partial maxima keep the reduction off one long chain
        float ex[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) ex[a] = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; c += 2) {
          tmem_ld32(lane_base + s_col + c * 32, va);
          tmem_ld32(lane_base + s_col + c * 32 + 32, vb);
          tmem_wait_ld();
          if (neg) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              va[i] = -va[i];
              vb[i] = -vb[i];
            }
          }
          if (!need_mask) {
#pragma unroll
            for (int i = 0; i < 32; ++i) ex[i & 7] = max3f(ex[i & 7], va[i], vb[i]);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              if (key0 + c * 32 + i <= limit) ex[i & 7] = fmaxf(ex[i & 7], va[i]);
              if (key0 + c * 32 + 32 + i <= limit) ex[i & 7] = fmaxf(ex[i & 7], vb[i]);
            }
          }
        }
        const float ext = fmaxf(fmaxf(fmaxf(ex[0], ex[1]), fmaxf(ex[2], ex[3])),
                                fmaxf(fmaxf(ex[4], ex[5]), fmaxf(ex[6], ex[7])));
        // a tile past the row's limit leaves the max at -inf and its P all zeros
        mx = ext == -INFINITY ? -INFINITY : ext * fabsf(p.scale_log2);
      }
      const bool resc = mx > m_used + kRescaleThreshold;
      if (__any_sync(0xffffffffu, resc)) {
        const float m_new = resc ? mx : m_used;
        const float alpha = ex2(m_used - m_new);  // 0 when m_used is -inf, 1 when unchanged
        if (j > 0) {
          // PV_{j-1} must be done before O is rescaled
          ok = __all_sync(0xffffffffu, pf_wait(o_done, (j - 1) & 1, abort_flag));
          if (!ok) break;
          tc_fence_after();
          const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tmem_ld32(lane_base + o_col + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; i += 2) f2_unpack(f2_mul(f2_pack(o[i], o[i + 1]), a2), o[i], o[i + 1]);
            tmem_st32(lane_base + o_col + c * 32, o);
          }
        }
        lsum *= alpha;
        m_used = m_new;
      }
      // pass 2: P = 2^(x - m_used) for 64 keys at a time, written over the
      // columns those keys' scores just vacated: bf16 hi of keys [64 g, 64 g + 64)
      // in columns [64 g, 64 g + 32), the bf16 residual lo in [64 g + 32, 64 g + 64),
      // two keys per column.
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        float va[32], vb[32];
        tmem_ld32(lane_base + s_col + 64 * g, va);
        tmem_ld32(lane_base + s_col + 64 * g + 32, vb);
        tmem_wait_ld();
        uint32_t hi[32], lo[32];
        // pairs of keys in packed f32x2 arithmetic: one FMA, one ADD and one
        // SUB instruction per two scores
        const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
        const uint64_t nm2 = f2_pack(-m_used, -m_used);
        uint64_t ls2[2] = {0ull, 0ull};  // independent partial row sums (pairs)
        if (!need_mask) {
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            const int kk = 2 * u;  // key within the group
            const float s0 = kk < 32 ? va[kk] : vb[kk - 32];
            const float s1 = kk < 32 ? va[kk + 1] : vb[kk - 31];
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(s0, s1), sc2, nm2), x0, x1);
            const float e0 = ex2(x0), e1 = ex2(x1);
            const uint64_t e = f2_pack(e0, e1);
            ls2[u & 1] = f2_add(ls2[u & 1], e);
            if constexpr (F16PV) {
              hi[u] = pack_f16x2_rn(e0, e1);
            } else {
              hi[u] = pack_bf16x2(e0, e1);
              float r0, r1;
              f2_unpack(f2_sub(e, f2_pack(bf16_lo_to_f32(hi[u]), bf16_hi_to_f32(hi[u]))), r0, r1);
              lo[u] = pack_bf16x2(r0, r1);
            }
          }
        } else {
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            const int kk = 2 * u;
            const float s0 = kk < 32 ? va[kk] : vb[kk - 32];
            const float s1 = kk < 32 ? va[kk + 1] : vb[kk - 31];
            const int key = key0 + 64 * g + kk;
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(s0, s1), sc2, nm2), x0, x1);
            const float e0 = key <= limit ? ex2(x0) : 0.f;
            const float e1 = key + 1 <= limit ? ex2(x1) : 0.f;
            const uint64_t e = f2_pack(e0, e1);
            ls2[u & 1] = f2_add(ls2[u & 1], e);
            if constexpr (F16PV) {
              hi[u] = pack_f16x2_rn(e0, e1);
            } else {
              hi[u] = pack_bf16x2(e0, e1);
              float r0, r1;
              f2_unpack(f2_sub(e, f2_pack(bf16_lo_to_f32(hi[u]), bf16_hi_to_f32(hi[u]))), r0, r1);
              lo[u] = pack_bf16x2(r0, r1);
            }
          }
        }
        {
          float a0, a1, b0, b1;
          f2_unpack(ls2[0], a0, a1);
          f2_unpack(ls2[1], b0, b1);
          lsum += (a0 + a1) + (b0 + b1);
        }
        tmem_st32u(lane_base + s_col + 64 * g, hi);
        if constexpr (!F16PV) tmem_st32u(lane_base + s_col + 64 * g + 32, lo);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (!ok) {
      if (lane == 0) pf_abort(abort_flag);
    } else {
      // epilogue: wait for the last PV, then out = O / l
      ok = __all_sync(0xffffffffu, pf_wait(o_done, (ntiles - 1) & 1, abort_flag));
      if (!ok) {
        if (lane == 0) pf_abort(abort_flag);
      } else {
        tc_fence_after();
        const float inv = p.out_scale / lsum;
        const size_t orow_idx = size_t(qs + tok) * p.q_heads + size_t(kvh) * G + head;
        float* orow = p.out + orow_idx * D;
        uint4* orow_bf16 = reinterpret_cast<uint4*>(
            reinterpret_cast<__nv_bfloat16*>(p.out) + orow_idx * D);
        if (p.lse && valid_row) p.lse[orow_idx] = m_used + __log2f(lsum);
        if (p.o_tma && !p.out_bf16 && __all_sync(0xffffffffu, valid_row)) {
          // The warp's 32 rows (32/G tokens x the G heads) in 32-column boxes
          // of 32 rows x 128 bytes, 128-byte swizzled, then one TMA store per
          // box.  Tile 0 stages over K stages 0-1, free once S_1 of the last
          // tile is done (before PV_0 of it); tile 1 over the next 128 rows'
          // worth, free once its own last PV -- the CTA's last MMA -- is done.
          const uint32_t stage = sbase + L::kKOff + uint32_t(wg) * (kPfRows * D * 4) +
                                 uint32_t(warp & 3) * (32 * D * 4);
          const uint32_t row_at = stage + uint32_t(lane) * 128;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tmem_ld32(lane_base + o_col + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 8; ++i)
              st_shared_f4(row_at + c * 4096 + ((uint32_t(i) ^ uint32_t(lane & 7)) << 4),
                           o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv,
                           o[4 * i + 3] * inv);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int tok0 = qs + t0 + wg * TPT + (warp & 3) * (32 / G);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) tma_store_3d(&tmap_o, stage + c * 4096, c * 32, kvh * G, tok0);
            bulk_commit_group();
            // shared memory is read before the item ends (the next item's
            // copies, or the next CTA, reuse it); the global writes finish
            // on their own
            bulk_wait_read_all();
          }
          __syncwarp();
        } else {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32(lane_base + o_col + c * 32, o);
          tmem_wait_ld();
          if (valid_row && p.out_bf16) {  // the same products, rounded to bf16
#pragma unroll
            for (int i = 0; i < 32; i += 8)
              orow_bf16[(c * 32 + i) / 8] = make_uint4(
                  pack_bf16x2(o[i] * inv, o[i + 1] * inv), pack_bf16x2(o[i + 2] * inv, o[i + 3] * inv),
                  pack_bf16x2(o[i + 4] * inv, o[i + 5] * inv), pack_bf16x2(o[i + 6] * inv, o[i + 7] * inv));
          } else if (valid_row) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4*>(orow + c * 32 + i) =
                  make_float4(o[i] * inv, o[i + 1] * inv, o[i + 2] * inv, o[i + 3] * inv);
          }
        }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

// Item `idx` of a launch (pairs x tiles items) -> its pair and query tile.
// Pair-major: a pair's tiles run back to back, longest first, so the CTAs
// resident at any time share the K/V of few pairs in L2 instead of touching
// every pair's pages at once; pairs go in seq_order (longest context first,
// which keeps the grid close to longest-first overall) when it is given.
// Returns false for an order entry outside the batch (the item is skipped).
__device__ __forceinline__ bool item_pair_tile(const PrefillParams& p, long long idx, int tiles,
                                               int& pair, int& tile) {
  const int pr = int(idx / tiles);
  tile = tiles - 1 - int(idx - (long long)pr * tiles);
  if (!p.seq_order) {
    pair = pr;
    return true;
  }
  const int rank = pr / p.kv_heads;
  const int seq = __ldg(p.seq_order + rank);
  pair = seq * p.kv_heads + (pr - rank * p.kv_heads);
  return seq >= 0 && seq < p.num_seqs;
}

}  // namespace pkv
