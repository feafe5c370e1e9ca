// Multi-query paged decode: K query tokens per sequence, each attending
// causally over the sequence's context -- the verification step of
// speculative decoding, where K drafted tokens are checked in one pass
// ("Cache KV, attention et optimisation de l'inference", section "Decodage
// speculatif": guess the next tokens cheaply, then verify them all at once).
//
// What is computed: for sequence s with context_len L (the K drafted tokens
// already appended) and query token t < K at position L - K + t, out[s, t, h]
// = softmax(q[s, t, h] . K_s[0 .. L-K+t]^T * scale) V_s[0 .. L-K+t] -- the
// chunked prefill of a K-token chunk with the bottom-right causal mask
// ("Optimisation de l'inference", "Etape 2"), GQA head h reading KV head h/G.
//
// Design (GB300): the bf16 decode kernel's structure with the query tokens of
// a sequence added to the MMA rows, so each K/V byte is still read from HBM
// once per (sequence, KV head) and the kernel stays bound by HBM:
//  * rows = K tokens x G heads of the group (token-major), padded to 16 x MT
//    (MT = 1 or 2 m16 tiles: up to 32 rows, e.g. K = 4 drafts at G = 8);
//  * Q is staged in shared memory (rows of D bf16, padded by 16 bytes so the
//    8 rows of an ldmatrix phase hit distinct banks) and loaded per k-step as
//    A fragments -- two m-tiles of Q in registers would not leave room for
//    two m-tiles of output accumulators;
//  * each row has its own causal limit L - K + t; only the last pages of a
//    sequence need the per-row mask;
//  * split-K partitions, per-warp TMA rings, the P hi + lo split, V zeroing of
//    rows past the length and the log-sum-exp merge are those of the decode.
#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_decode_common.cuh"

namespace pkv {

static __device__ unsigned g_verify_error = 0;

constexpr int kVerifyWarps = 4;
constexpr int kVerifyStages = 3;
constexpr int kVerifyMaxPartitionBlocks = 1024;

template <int D, int MT>
struct VerifyTile {
  static constexpr int kRows = 16 * MT;
  static constexpr int kHalfBytes = kBlockTokens * 128;       // 16 rows x 64 bf16
  static constexpr int kTileBytes = kBlockTokens * D * 2;     // one block, one head
  static constexpr int kStageBytes = 2 * kTileBytes;          // K + V
  static constexpr int kRingBytes = kVerifyStages * kStageBytes;
  static constexpr int kRingsBytes = kVerifyWarps * kRingBytes;
  static constexpr int kBarOffset = kRingsBytes;
  static constexpr int kIdsOffset = kBarOffset + kVerifyWarps * kVerifyStages * 8;
  static constexpr int kQStride = D * 2 + 16;                 // bytes per staged Q row
  static constexpr int kQOffset = kIdsOffset + kVerifyMaxPartitionBlocks * 4;
  static constexpr int kSmemBytes = kQOffset + kRows * kQStride + 1024;  // +align slack
  // the cross-warp merge reuses each warp's ring: [rows][D] outputs + m, l
  static_assert(kRows * D * 4 + 2 * kRows * 4 <= kRingBytes, "merge does not fit the ring");
};

struct VerifyParams {
  DecodeParams d;  // rows of q / out: (seq * q_len + t) * q_heads + head
  int q_len;
};

template <int D, int G, int MT>
__global__ void __launch_bounds__(kVerifyWarps * 32, 2)
paged_verify_kernel(const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v, const VerifyParams vp) {
  griddep_wait();  // inputs may have been written by the previous kernel in the stream
  using T = VerifyTile<D, MT>;
  const DecodeParams& p = vp.d;
  constexpr int R = T::kRows;
  constexpr int KSTEPS = D / 16;  // k-steps of QK^T
  constexpr int NT = D / 8;       // n-tiles of the output
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  int32_t* ids = reinterpret_cast<int32_t*>(smem + T::kIdsOffset);
  uint8_t* qs = smem + T::kQOffset;

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  const int pair = blockIdx.x;
  const int part = blockIdx.y;
  const int seq = pair / p.kv_heads;
  const int kvh = pair - seq * p.kv_heads;
  const int K = vp.q_len;
  const int rows_used = G * K;  // <= R (checked on the host)

  const SeqSpan sp = seq_span(__ldg(p.context_lens + seq), p, seq);
  const int len = sp.len;
  if (part == 0 && threadIdx.x == 0) {
    if (sp.bad) atomicOr(&g_verify_error, kErrBadContext);
    if (len < K) atomicOr(&g_verify_error, kErrBadQueryRange);  // tokens before position 0
  }
  const int nparts_s = span_parts(sp, p);
  if (part >= nparts_s) return;
  // output row of local row r = t * G + h
  auto out_row = [&](int r) {
    const int t = r / G, h = r - (r / G) * G;
    return (size_t(seq) * K + t) * p.q_heads + size_t(kvh) * G + h;
  };
  if (sp.count == 0) {  // empty context: zeros
    for (int i = threadIdx.x; i < rows_used * D; i += blockDim.x)
      store_out(p, out_row(i / D) * D + (i - (i / D) * D), 0.f);
    return;
  }
  const int b0 = sp.first + part * p.partition_blocks;  // first block of this partition
  const int nb_local = min(sp.first + sp.count - b0, p.partition_blocks);

  // Stage this partition's block ids (ids outside the pool are flagged; their
  // TMA boxes are out of bounds and read as zeros) and the Q rows.
  const int32_t* table = p.block_tables + size_t(seq) * p.max_blocks_per_seq + b0;
  for (int i = threadIdx.x; i < nb_local; i += blockDim.x) {
    const int32_t id = __ldg(table + i);
    if (id < 0 || id >= p.num_blocks) atomicOr(&g_verify_error, kErrBadBlockId);
    ids[i] = id;
  }
  constexpr int kVecPerRow = D / 8;  // 16-byte vectors of bf16
  for (int i = threadIdx.x; i < R * kVecPerRow; i += blockDim.x) {
    const int r = i / kVecPerRow, c = i - r * kVecPerRow;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r < rows_used) v = __ldg(reinterpret_cast<const uint4*>(p.q + out_row(r) * D) + c);
    *reinterpret_cast<uint4*>(qs + r * T::kQStride + c * 16) = v;
  }
  const uint32_t ring = smem_u32(smem + warp * T::kRingBytes);
  const uint32_t bars = smem_u32(smem + T::kBarOffset) + warp * kVerifyStages * 8;
  if (lane == 0) {
    for (int st = 0; st < kVerifyStages; ++st) mbar_init(bars + st * 8, 1);
    fence_barrier_init();
  }
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_v);
  }
  __syncthreads();  // ids and Q staged, barriers initialised

  const int cnt = warp < nb_local ? (nb_local - warp + kVerifyWarps - 1) / kVerifyWarps : 0;
  auto issue = [&](int i) {
    const int st = i % kVerifyStages;
    const uint32_t bar = bars + st * 8;
    const uint32_t kdst = ring + st * T::kStageBytes;
    const uint32_t vdst = kdst + T::kTileBytes;
    const int bid = ids[warp + i * kVerifyWarps];
    mbar_arrive_expect_tx(bar, T::kStageBytes);
#pragma unroll
    for (int h = 0; h < D / 64; ++h) {
      tma_load_4d(kdst + h * T::kHalfBytes, &tmap_k, bar, h * 64, kvh, 0, bid);
      tma_load_4d(vdst + h * T::kHalfBytes, &tmap_v, bar, h * 64, kvh, 0, bid);
    }
  };
  if (lane == 0) {
    for (int i = 0; i < cnt && i < kVerifyStages; ++i) issue(i);
  }
  int issued = cnt < kVerifyStages ? cnt : kVerifyStages;

  // Per-lane ldmatrix geometry: K and V as in the decode; Q rows for the A
  // fragments (matrices: rows 0-7 | 8-15 x k 0-7 | 8-15).
  const int mi = lane >> 3, mr = lane & 7;
  const int k_tok = (mi >> 1) * 8 + mr;
  const int v_tok = (mi & 1) * 8 + mr;
  const uint32_t q_lane =
      smem_u32(qs) + ((lane & 7) + ((lane >> 3) & 1) * 8) * T::kQStride + (lane >> 4) * 16;

  // Causal limit (last key index seen) of this lane's rows mt * 16 + gid + 8 hf;
  // padding rows take the last token's limit.
  int lim[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int t = min((mt * 16 + gid + 8 * hf) / G, K - 1);
      lim[mt][hf] = len - K + t;
    }
  const int first_masked = len - K + 1;  // keys from here on are past some row's limit

  float o[MT][NT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int n = 0; n < NT; ++n) o[mt][n][0] = o[mt][n][1] = o[mt][n][2] = o[mt][n][3] = 0.f;
  float m[MT][2], l[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) m[mt][0] = m[mt][1] = -INFINITY, l[mt][0] = l[mt][1] = 0.f;
  bool failed = false;
  int i = 0;
  for (; i < cnt; ++i) {
    const int st = i % kVerifyStages;
    const uint32_t par = (i / kVerifyStages) & 1;
    const bool ready = __all_sync(0xffffffffu, mbar_wait_bounded(bars + st * 8, par));
    if (!ready) {
      failed = true;
      break;
    }
    const uint32_t kbase = ring + st * T::kStageBytes;
    const uint32_t vbase = kbase + T::kTileBytes;
    const int tok0 = (b0 + warp + i * kVerifyWarps) * kBlockTokens;

    // S = Q K^T for 16 keys (two n-tiles of 8) and every m-tile.
    float s[MT][2][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) s[mt][nt][0] = s[mt][nt][1] = s[mt][nt][2] = s[mt][nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      const int chunk = 2 * kk + (mi & 1);
      const uint32_t addr = kbase + (chunk >> 3) * T::kHalfBytes + k_tok * 128 +
                            (((chunk & 7) ^ (k_tok & 7)) << 4);
      uint32_t b0r, b1r, b2r, b3r;
      ldsm_x4(addr, b0r, b1r, b2r, b3r);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(q_lane + mt * 16 * T::kQStride + kk * 32, a0, a1, a2, a3);
        mma_bf16_16816(s[mt][0], a0, a1, a2, a3, b0r, b1r);
        mma_bf16_16816(s[mt][1], a0, a1, a2, a3, b2r, b3r);
      }
    }

    // Online softmax in the log2 domain with each row's causal limit.
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[mt][nt][e] *= p.scale_log2;
    if (tok0 + kBlockTokens > first_masked) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (tok0 + nt * 8 + tig * 2 + (e & 1) > lim[mt][e >> 1]) s[mt][nt][e] = -INFINITY;
    }
    uint32_t ph[MT][4], pl[MT][4];
    bool rescale = false;
    float alpha[MT][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      float pr[2][4];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float mx = fmaxf(fmaxf(s[mt][0][2 * hf], s[mt][0][2 * hf + 1]),
                         fmaxf(s[mt][1][2 * hf], s[mt][1][2 * hf + 1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float mn = fmaxf(m[mt][hf], mx);
        // a row that has seen no key yet keeps max -inf: exponentiate against 0
        const float mref = mn == -INFINITY ? 0.f : mn;
        alpha[mt][hf] = ex2(m[mt][hf] - mref);
        rescale |= alpha[mt][hf] != 1.f;
        m[mt][hf] = mn;
        pr[0][2 * hf] = ex2(s[mt][0][2 * hf] - mref);
        pr[0][2 * hf + 1] = ex2(s[mt][0][2 * hf + 1] - mref);
        pr[1][2 * hf] = ex2(s[mt][1][2 * hf] - mref);
        pr[1][2 * hf + 1] = ex2(s[mt][1][2 * hf + 1] - mref);
        l[mt][hf] = l[mt][hf] * alpha[mt][hf] + (pr[0][2 * hf] + pr[0][2 * hf + 1]) +
                    (pr[1][2 * hf] + pr[1][2 * hf + 1]);
      }
      // P as the A operand (rows, k = 16 keys), split into bf16 hi + lo.
      ph[mt][0] = pack_bf16x2(pr[0][0], pr[0][1]);
      ph[mt][1] = pack_bf16x2(pr[0][2], pr[0][3]);
      ph[mt][2] = pack_bf16x2(pr[1][0], pr[1][1]);
      ph[mt][3] = pack_bf16x2(pr[1][2], pr[1][3]);
      pl[mt][0] = pack_bf16x2(pr[0][0] - bf16_lo_to_f32(ph[mt][0]), pr[0][1] - bf16_hi_to_f32(ph[mt][0]));
      pl[mt][1] = pack_bf16x2(pr[0][2] - bf16_lo_to_f32(ph[mt][1]), pr[0][3] - bf16_hi_to_f32(ph[mt][1]));
      pl[mt][2] = pack_bf16x2(pr[1][0] - bf16_lo_to_f32(ph[mt][2]), pr[1][1] - bf16_hi_to_f32(ph[mt][2]));
      pl[mt][3] = pack_bf16x2(pr[1][2] - bf16_lo_to_f32(ph[mt][3]), pr[1][3] - bf16_hi_to_f32(ph[mt][3]));
    }
    // rescale the accumulators only when some row's max moved
    if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          o[mt][n][0] *= alpha[mt][0];
          o[mt][n][1] *= alpha[mt][0];
          o[mt][n][2] *= alpha[mt][1];
          o[mt][n][3] *= alpha[mt][1];
        }
    }

    // Keys past the length may hold anything (NaN included): zero their V so
    // that their zero weights give exactly 0.
    uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
    if (tok0 + kBlockTokens > len) {
      const int k0 = tok0 + 2 * tig;
      vm0 = (k0 < len ? 0x0000ffffu : 0u) | (k0 + 1 < len ? 0xffff0000u : 0u);
      vm1 = (k0 + 8 < len ? 0x0000ffffu : 0u) | (k0 + 9 < len ? 0xffff0000u : 0u);
    }
    // O += P V: V tiles through ldmatrix.trans (B operand, k = keys, n = dims).
#pragma unroll
    for (int dn = 0; dn < D / 16; ++dn) {
      const int chunk = 2 * dn + (mi >> 1);
      const uint32_t addr = vbase + (chunk >> 3) * T::kHalfBytes + v_tok * 128 +
                            (((chunk & 7) ^ (v_tok & 7)) << 4);
      uint32_t b0r, b1r, b2r, b3r;
      ldsm_x4_trans(addr, b0r, b1r, b2r, b3r);
      b0r &= vm0;
      b1r &= vm1;
      b2r &= vm0;
      b3r &= vm1;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        mma_bf16_16816(o[mt][2 * dn], ph[mt][0], ph[mt][1], ph[mt][2], ph[mt][3], b0r, b1r);
        mma_bf16_16816(o[mt][2 * dn + 1], ph[mt][0], ph[mt][1], ph[mt][2], ph[mt][3], b2r, b3r);
        mma_bf16_16816(o[mt][2 * dn], pl[mt][0], pl[mt][1], pl[mt][2], pl[mt][3], b0r, b1r);
        mma_bf16_16816(o[mt][2 * dn + 1], pl[mt][0], pl[mt][1], pl[mt][2], pl[mt][3], b2r, b3r);
      }
    }

    __syncwarp();  // every lane is done reading this stage
    if (i + kVerifyStages < cnt) {
      if (lane == 0) issue(i + kVerifyStages);
      ++issued;
    }
  }

  if (failed) {
    // Record the timeout and wait (bounded) for this warp's copies still in
    // flight, so no TMA writes into shared memory after the CTA exits.
    if (lane == 0) {
      atomicOr(&g_verify_error, kErrWaitTimeout);
      for (int k = i; k < issued; ++k)
        (void)mbar_wait_bounded(bars + (k % kVerifyStages) * 8, (k / kVerifyStages) & 1);
    }
    __syncwarp();
  }

  // Row sums were kept per lane: reduce over the quad.
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      l[mt][hf] += __shfl_xor_sync(0xffffffffu, l[mt][hf], 1);
      l[mt][hf] += __shfl_xor_sync(0xffffffffu, l[mt][hf], 2);
    }

  // Cross-warp merge through shared memory (each warp reuses its own ring).
  float* mo = reinterpret_cast<float*>(smem + warp * T::kRingBytes);  // [R][D]
  float* mml = mo + R * D;                                            // m[R], l[R]
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int r = mt * 16 + gid + 8 * hf;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        mo[r * D + n * 8 + tig * 2] = o[mt][n][2 * hf];
        mo[r * D + n * 8 + tig * 2 + 1] = o[mt][n][2 * hf + 1];
      }
      if (tig == 0) {
        mml[r] = m[mt][hf];
        mml[R + r] = l[mt][hf];
      }
    }
  __syncthreads();

  const bool final_out = (nparts_s == 1) && !p.force_partials;
  for (int idx = threadIdx.x; idx < rows_used * D; idx += blockDim.x) {
    const int row = idx / D, col = idx - row * D;
    float big = -INFINITY;
#pragma unroll
    for (int w = 0; w < kVerifyWarps; ++w) {
      const float* wm = reinterpret_cast<const float*>(smem + w * T::kRingBytes) + R * D;
      big = fmaxf(big, wm[row]);
    }
    // a row that saw no key in this partition (its limit lies before it)
    const float bref = big == -INFINITY ? 0.f : big;
    float tot = 0.f, val = 0.f;
#pragma unroll
    for (int w = 0; w < kVerifyWarps; ++w) {
      const float* wo = reinterpret_cast<const float*>(smem + w * T::kRingBytes);
      const float wgt = ex2(wo[R * D + row] - bref);
      tot += wo[R * D + R + row] * wgt;
      val += wo[row * D + col] * wgt;
    }
    const float res = tot > 0.f ? val / tot : 0.f;
    const size_t orow = out_row(row);
    if (final_out) {
      store_out(p, orow * D + col, res);
    } else {
      const size_t prow = orow * p.num_parts + part;
      p.part_o[prow * D + col] = res;
      if (col == 0) p.part_lse[prow] = tot > 0.f ? big + __log2f(tot) : -INFINITY;
    }
  }
}

// Device address of this unit's error word on the current device.
cudaError_t verify_error_word(unsigned** word) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(word), g_verify_error);
}

unsigned read_verify_error(bool clear) {
  unsigned word = 0;
  if (cudaMemcpyFromSymbol(&word, g_verify_error, sizeof(word)) != cudaSuccess) return ~0u;
  if (clear) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_verify_error, &zero, sizeof(zero)) != cudaSuccess) return ~0u;
  }
  return word;
}

template <int D, int G, int MT>
static cudaError_t launch_verify_t(const VerifyParams& vp, int num_seqs, const CUtensorMap* tk,
                                   const CUtensorMap* tv, cudaStream_t stream) {
  using T = VerifyTile<D, MT>;
  static std::atomic<int> attr_done[kAttrMaxDevices];
  {
    const cudaError_t e =
        set_smem_limit_once(paged_verify_kernel<D, G, MT>, T::kSmemBytes, attr_done);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(num_seqs * vp.d.kv_heads, vp.d.num_parts);
  cudaError_t e = launch_after_previous(paged_verify_kernel<D, G, MT>, grid,
                                        dim3(kVerifyWarps * 32), T::kSmemBytes, stream, *tk, *tv,
                                        vp);
  if (e != cudaSuccess) return e;
  // The merge sees the K tokens of a sequence as K x q_heads rows of it.
  DecodeParams mp = vp.d;
  mp.q_heads = vp.d.q_heads * vp.q_len;
  return launch_decode_merge(mp, num_seqs, D, stream);
}

template <int D, int MT>
static cudaError_t launch_verify_m(const VerifyParams& vp, int num_seqs, int group,
                                   const CUtensorMap* tk, const CUtensorMap* tv,
                                   cudaStream_t st) {
  switch (group) {
    case 1: return launch_verify_t<D, 1, MT>(vp, num_seqs, tk, tv, st);
    case 2: return launch_verify_t<D, 2, MT>(vp, num_seqs, tk, tv, st);
    case 4: return launch_verify_t<D, 4, MT>(vp, num_seqs, tk, tv, st);
    case 8: return launch_verify_t<D, 8, MT>(vp, num_seqs, tk, tv, st);
    case 16: return launch_verify_t<D, 16, MT>(vp, num_seqs, tk, tv, st);
    default: return cudaErrorInvalidValue;
  }
}

int verify_max_rows() { return 32; }

cudaError_t launch_paged_verify(const DecodeArgs& a, int q_len, const CUtensorMap* tmap_k,
                                const CUtensorMap* tmap_v, cudaStream_t stream) {
  VerifyParams vp;
  DecodeParams& prm = vp.d;
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
  prm.out_bf16 = a.out_bf16 ? 1 : 0;
  prm.first_block = 0;
  prm.force_partials = 0;
  prm.extra_o = nullptr;
  prm.extra_lse = nullptr;
  vp.q_len = q_len;
  const int group = a.q_heads / a.kv_heads;
  const int rows = group * q_len;
  if (q_len <= 0 || rows > verify_max_rows()) return cudaErrorInvalidValue;
  const bool two = rows > 16;
  if (a.d_head == 128)
    return two ? launch_verify_m<128, 2>(vp, a.num_seqs, group, tmap_k, tmap_v, stream)
               : launch_verify_m<128, 1>(vp, a.num_seqs, group, tmap_k, tmap_v, stream);
  if (a.d_head == 64)
    return two ? launch_verify_m<64, 2>(vp, a.num_seqs, group, tmap_k, tmap_v, stream)
               : launch_verify_m<64, 1>(vp, a.num_seqs, group, tmap_k, tmap_v, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
