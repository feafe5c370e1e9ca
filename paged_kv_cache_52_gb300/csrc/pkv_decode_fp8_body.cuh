// The per-page body of the decode over an FP8 (e4m3) cache, shared by the
// split kernel (paged_decode_fp8.cu) and the flat split
// (paged_decode_flat.cu): the f16 warp MMAs on converted codes, the online
// softmax and P V for one or two landed pages of one warp's ring.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "pkv_decode_common.cuh"
#include "pkv_device.cuh"

namespace pkv {

constexpr int kF8D = 128;
constexpr unsigned kErrFp16Range = 1u << 6;

// One ring stage: a page of one KV head, K codes then V codes.
struct F8Page {
  static constexpr int kTileBytes = kBlockTokens * kF8D;  // 16 keys x 128 codes
  static constexpr int kStageBytes = 2 * kTileBytes;      // K + V
};

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four e4m3 codes (byte i = code i) -> two f16x2: codes 0, 1 in `lo`, codes
// 2, 3 in `hi` (first code in the low half); the conversion is exact.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t codes, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\t"
      "mov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(codes));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Two bf16 (one 32-bit word) -> f16x2, flagging values outside f16's range.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w, bool* range_ok) {
  const float a = bf16_lo_to_f32(w), b = bf16_hi_to_f32(w);
  if (!(fabsf(a) < 65520.f) || !(fabsf(b) < 65520.f)) *range_ok = false;
  return pack_f16x2(a, b);
}

// An 8x8 matrix of 16-bit values held one row per lane quad (lane l: row
// l / 4, columns 2 (l % 4), 2 (l % 4) + 1) -> the same fragment of its transpose.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// Running state of one warp: O^T accumulators (m-tile mt, row gid = dim
// 16 mt + 2 gid, row gid + 8 = dim 16 mt + 2 gid + 1; columns 2 tig, 2 tig + 1
// = heads of n-tile nh), and the running max and this lane's part of the sum
// of heads 8 nh + 2 tig + c.
template <int G>
struct F8Acc {
  static constexpr int NH = (G + 7) / 8;
  static constexpr int MT = kF8D / 16;
  float o[NH][MT][4];
  float m[NH][2], l[NH][2];
};

// NP consecutive pages of this warp (ring slots i, i + 1, ...), all landed.
// Two pages per call keep two independent MMA and exponential chains in
// flight and share one max reduction and one rescale among 32 keys.
// STAGES: ring stages (page i in slot i % STAGES); PAGE_STRIDE: the second
// page's position, in pages after the first (the warps of a split CTA take
// every PAGE_STRIDE-th page; a flat warp takes consecutive ones).
template <int G, int NP, int STAGES, int PAGE_STRIDE>
__device__ __forceinline__ void fp8_pages(F8Acc<G>& A, const uint32_t (&qf)[(G + 7) / 8][8][2],
                                          uint32_t ring, int i, int tok_first, int len,
                                          float scale_log2, int lane) {
  using T = F8Page;
  constexpr int NH = F8Acc<G>::NH;
  constexpr int MT = F8Acc<G>::MT;
  const int gid = lane >> 2, tig = lane & 3;
  const int mi = lane >> 3, mr = lane & 7;
  const int k_tok = (mi >> 1) * 8 + mr;  // K: matrices (keys 0-7|8-15) x (chunk even|odd)
  const int v_tok = (mi & 1) * 8 + mr;   // V: matrices (keys 0-7|8-15) x (chunk even|odd)
  uint32_t kbase[NP];
  int tok0[NP];
#pragma unroll
  for (int pg = 0; pg < NP; ++pg) {
    kbase[pg] = ring + ((i + pg) % STAGES) * T::kStageBytes;
    tok0[pg] = tok_first + pg * PAGE_STRIDE * kBlockTokens;
  }

  // S^T = K Q^T: one ldmatrix.x4 covers two k-steps of both 8-key halves:
  // a lane gets 4 consecutive dims of key gid (r0 | r1) and of key gid + 8
  // (r2 | r3).  Even and odd k-steps accumulate separately.
  float s[NP][NH][4], s_odd[NP][NH][4];
#pragma unroll
  for (int pg = 0; pg < NP; ++pg)
#pragma unroll
    for (int nh = 0; nh < NH; ++nh)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[pg][nh][e] = s_odd[pg][nh][e] = 0.f;
#pragma unroll
  for (int kp = 0; kp < 4; ++kp) {
#pragma unroll
    for (int pg = 0; pg < NP; ++pg) {
      const int chunk = 2 * kp + (mi & 1);
      uint32_t r0, r1, r2, r3;
      ldsm_x4(kbase[pg] + k_tok * 128 + (((chunk ^ (k_tok & 7))) << 4), r0, r1, r2, r3);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t a0, a1, a2, a3;
        e4m3x4_to_f16x2x2(h ? r1 : r0, a0, a2);  // key gid
        e4m3x4_to_f16x2x2(h ? r3 : r2, a1, a3);  // key gid + 8
#pragma unroll
        for (int nh = 0; nh < NH; ++nh)
          mma_f16_16816(h ? s_odd[pg][nh] : s[pg][nh], a0, a1, a2, a3, qf[nh][2 * kp + h][0],
                        qf[nh][2 * kp + h][1]);
      }
    }
  }

  // Online softmax in the log2 domain (k_scale folded into scale_log2), per
  // head column over the pages' keys (rows: this lane's gid and gid + 8 of
  // each page, the other keys in the lanes with the same tig).
  bool k0_in[NP], k1_in[NP];
#pragma unroll
  for (int pg = 0; pg < NP; ++pg) {
    k0_in[pg] = tok0[pg] + gid < len;
    k1_in[pg] = tok0[pg] + gid + 8 < len;
  }
  uint32_t pb[NP][NH][2];
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
    // P^T as the B operand of the P V product: k = a page's keys, n = the
    // heads; the lane's (key, two heads) pairs transposed into (two keys, head)
#pragma unroll
    for (int pg = 0; pg < NP; ++pg) {
      pb[pg][nh][0] = movmatrix_trans(pack_f16x2(pr[pg][0], pr[pg][1]));  // keys 2 tig, +1
      pb[pg][nh][1] = movmatrix_trans(pack_f16x2(pr[pg][2], pr[pg][3]));  // keys 8 + 2 tig, +1
    }
  }
  // After the first pages the running max rarely moves: skip the rescale
  // (alpha = 1 exactly) unless some head of the warp needs it.
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

  // O^T += V^T P^T.  ldmatrix.trans over the codes as 16-bit units gives a
  // lane keys (2 tig, 2 tig + 1) x dims (2 gid, 2 gid + 1) of a 16-dim
  // chunk; the byte permute splits that into the key pair of dim 2 gid (row
  // gid) and of dim 2 gid + 1 (row gid + 8).
  // Rows of the last page past the length may hold any code, NaN included:
  // zero them (their P is 0).  Each 16-bit unit holds one key's two codes,
  // keys (2 tig, 2 tig + 1) in r0 / r2 and 8 more in r1 / r3.
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
#pragma unroll
  for (int cp = 0; cp < 4; ++cp) {
#pragma unroll
    for (int pg = 0; pg < NP; ++pg) {
      const int chunk = 2 * cp + (mi >> 1);
      uint32_t r0, r1, r2, r3;
      ldsm_x4_trans(kbase[pg] + T::kTileBytes + v_tok * 128 + (((chunk ^ (v_tok & 7))) << 4), r0,
                    r1, r2, r3);
      r0 &= vm0[pg];
      r1 &= vm1[pg];
      r2 &= vm0[pg];
      r3 &= vm1[pg];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        // bytes (k0 d0, k0 d1, k1 d0, k1 d1) -> (k0 d0, k1 d0, k0 d1, k1 d1)
        uint32_t a0, a1, a2, a3;
        e4m3x4_to_f16x2x2(__byte_perm(h ? r2 : r0, 0u, 0x3120), a0, a1);  // keys 2 tig, +1
        e4m3x4_to_f16x2x2(__byte_perm(h ? r3 : r1, 0u, 0x3120), a2, a3);  // keys 8 + 2 tig, +1
#pragma unroll
        for (int nh = 0; nh < NH; ++nh)
          mma_f16_16816(A.o[nh][2 * cp + h], a0, a1, a2, a3, pb[pg][nh][0], pb[pg][nh][1]);
      }
    }
  }
}

}  // namespace pkv
