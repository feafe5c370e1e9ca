// KV append: scatter new K/V token rows into the paged pools through the
// per-token slot mapping (nano-vLLM page, section "Ecriture dans le cache":
// slot -1 skips the token, otherwise the row lands in block slot / 16 at
// offset slot % 16).
//
// One warp copies one token row of K and of V with 16-byte vector loads and
// stores; the grid strides over tokens.  Pure HBM copy: 2 * row bytes read and
// 2 * row bytes written per token.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

static __device__ unsigned g_append_error = 0;

constexpr int kAppendThreads = 256;
constexpr int kAppendVecPerLane = 4;  // 16-byte vectors kept in flight per lane per row

// Checked append, first pass: one bit per slot of the pool (zeroed before).
// A token whose slot bit was already set shares its slot with an earlier
// token of the call: the mapping is rejected (*reject = 1), the error word
// records it, and the append that follows on the stream writes nothing.
// Slots -1 and outside the pool are left to the append (skipped there).
__global__ void __launch_bounds__(kAppendThreads)
slot_duplicates_kernel(const int64_t* __restrict__ slot_mapping, int64_t num_tokens,
                       int64_t num_slots, unsigned* __restrict__ bitmap, int* __restrict__ reject) {
  const int64_t stride = int64_t(gridDim.x) * kAppendThreads;
  for (int64_t t = int64_t(blockIdx.x) * kAppendThreads + threadIdx.x; t < num_tokens;
       t += stride) {
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0 || slot >= num_slots) continue;
    const unsigned bit = 1u << unsigned(slot & 31);
    if (atomicOr(bitmap + (slot >> 5), bit) & bit) {
      atomicOr(&g_append_error, kErrDuplicateSlot);
      atomicExch(reject, 1);
    }
  }
}

__global__ void __launch_bounds__(kAppendThreads)
kv_append_kernel(const uint4* __restrict__ k, int64_t k_stride_vec, const uint4* __restrict__ v,
                 int64_t v_stride_vec, const int64_t* __restrict__ slot_mapping,
                 int64_t num_tokens, uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                 int64_t num_slots, int row_vec, const int* __restrict__ reject,
                 int trigger_dependents) {
  // a decode step's attention may start beside this append: it waits for it
  // only where it reads the appended rows
  if (trigger_dependents) griddep_launch_dependents();
  if (reject && *reject) return;  // checked append of a mapping with a repeated slot
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t(blockIdx.x) * kAppendThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * kAppendThreads) >> 5;
  for (int64_t t = warp; t < num_tokens; t += nwarps) {
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot == -1) continue;
    if (slot < -1 || slot >= num_slots) {
      if (lane == 0) atomicOr(&g_append_error, kErrBadSlot);
      continue;
    }
    const uint4* ks = k + t * k_stride_vec;
    const uint4* vs = v + t * v_stride_vec;
    uint4* kd = k_cache + slot * row_vec;
    uint4* vd = v_cache + slot * row_vec;
    for (int base = 0; base < row_vec; base += 32 * kAppendVecPerLane) {
      uint4 kr[kAppendVecPerLane], vr[kAppendVecPerLane];
#pragma unroll
      for (int u = 0; u < kAppendVecPerLane; ++u) {
        const int i = base + u * 32 + lane;
        if (i < row_vec) {
          kr[u] = __ldg(ks + i);
          vr[u] = __ldg(vs + i);
        }
      }
#pragma unroll
      for (int u = 0; u < kAppendVecPerLane; ++u) {
        const int i = base + u * 32 + lane;
        if (i < row_vec) {
          kd[i] = kr[u];
          vd[i] = vr[u];
        }
      }
    }
  }
}

// Device address of this unit's error word on the current device.
cudaError_t append_error_word(unsigned** word) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(word), g_append_error);
}

unsigned read_append_error(bool clear) {
  unsigned word = 0;
  if (cudaMemcpyFromSymbol(&word, g_append_error, sizeof(word)) != cudaSuccess) return ~0u;
  if (clear) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_append_error, &zero, sizeof(zero)) != cudaSuccess) return ~0u;
  }
  return word;
}

cudaError_t launch_slot_duplicates(const int64_t* slot_mapping, int64_t num_tokens,
                                   int64_t num_slots, unsigned* bitmap, int* reject,
                                   cudaStream_t stream, int num_sms) {
  const int64_t blocks_needed = (num_tokens + kAppendThreads - 1) / kAppendThreads;
  const int64_t max_blocks = int64_t(num_sms) * 8;
  const int grid = int(blocks_needed < max_blocks ? blocks_needed : max_blocks);
  slot_duplicates_kernel<<<grid, kAppendThreads, 0, stream>>>(slot_mapping, num_tokens,
                                                              num_slots, bitmap, reject);
  return cudaGetLastError();
}

cudaError_t launch_kv_append(const void* k, int64_t k_stride, const void* v, int64_t v_stride,
                             const int64_t* slot_mapping, int64_t num_tokens, void* k_cache,
                             void* v_cache, int64_t num_slots, int row_elems,
                             cudaStream_t stream, int num_sms, const int* reject,
                             bool trigger_dependents) {
  const int row_vec = row_elems / 8;  // 8 bf16 per 16-byte vector
  const int64_t warps_needed = num_tokens;
  const int64_t blocks_needed = (warps_needed * 32 + kAppendThreads - 1) / kAppendThreads;
  const int64_t max_blocks = int64_t(num_sms) * 8;
  const int grid = int(blocks_needed < max_blocks ? blocks_needed : max_blocks);
  kv_append_kernel<<<grid, kAppendThreads, 0, stream>>>(
      static_cast<const uint4*>(k), k_stride / 8, static_cast<const uint4*>(v), v_stride / 8,
      slot_mapping, num_tokens, static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
      num_slots, row_vec, reject, trigger_dependents ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace pkv

// ---------------------------------------------------------------------------
// FP8 (e4m3) append: each element is quantized as float32(x) * inv_scale,
// rounded to nearest even with finite overflow saturating to +-448, and the
// code stored as one byte.  One warp per token; a lane converts 16 bf16 (two
// 16-byte loads) into 16 codes (one 16-byte store).
// ---------------------------------------------------------------------------
#include <cuda_fp8.h>

namespace pkv {

__device__ __forceinline__ uint32_t quant4_e4m3(uint2 bf4, float inv) {
  const float f0 = bf16_lo_to_f32(bf4.x) * inv, f1 = bf16_hi_to_f32(bf4.x) * inv;
  const float f2 = bf16_lo_to_f32(bf4.y) * inv, f3 = bf16_hi_to_f32(bf4.y) * inv;
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(f0, f1), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(f2, f3), __NV_SATFINITE, __NV_E4M3);
  return (lo & 0xffffu) | (hi << 16);
}

__global__ void __launch_bounds__(kAppendThreads)
kv_append_fp8_kernel(const uint4* __restrict__ k, int64_t k_stride_vec, const uint4* __restrict__ v,
                     int64_t v_stride_vec, const int64_t* __restrict__ slot_mapping,
                     int64_t num_tokens, uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                     int64_t num_slots, int row_vec16, float k_inv, float v_inv) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t(blockIdx.x) * kAppendThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * kAppendThreads) >> 5;
  for (int64_t t = warp; t < num_tokens; t += nwarps) {
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot == -1) continue;
    if (slot < -1 || slot >= num_slots) {
      if (lane == 0) atomicOr(&g_append_error, kErrBadSlot);
      continue;
    }
    const uint4* ks = k + t * k_stride_vec;  // 8 bf16 per vector
    const uint4* vs = v + t * v_stride_vec;
    uint4* kd = k_cache + slot * row_vec16;   // 16 codes per vector
    uint4* vd = v_cache + slot * row_vec16;
    for (int i = lane; i < row_vec16; i += 32) {
      const uint4 ka = __ldg(ks + 2 * i), kb = __ldg(ks + 2 * i + 1);
      const uint4 va = __ldg(vs + 2 * i), vb = __ldg(vs + 2 * i + 1);
      kd[i] = make_uint4(quant4_e4m3(make_uint2(ka.x, ka.y), k_inv),
                         quant4_e4m3(make_uint2(ka.z, ka.w), k_inv),
                         quant4_e4m3(make_uint2(kb.x, kb.y), k_inv),
                         quant4_e4m3(make_uint2(kb.z, kb.w), k_inv));
      vd[i] = make_uint4(quant4_e4m3(make_uint2(va.x, va.y), v_inv),
                         quant4_e4m3(make_uint2(va.z, va.w), v_inv),
                         quant4_e4m3(make_uint2(vb.x, vb.y), v_inv),
                         quant4_e4m3(make_uint2(vb.z, vb.w), v_inv));
    }
  }
}

cudaError_t launch_kv_append_fp8(const void* k, int64_t k_stride, const void* v, int64_t v_stride,
                                 const int64_t* slot_mapping, int64_t num_tokens, void* k_cache,
                                 void* v_cache, int64_t num_slots, int row_elems, float k_inv,
                                 float v_inv, cudaStream_t stream, int num_sms) {
  const int64_t blocks_needed = (num_tokens * 32 + kAppendThreads - 1) / kAppendThreads;
  const int64_t max_blocks = int64_t(num_sms) * 8;
  const int grid = int(blocks_needed < max_blocks ? blocks_needed : max_blocks);
  kv_append_fp8_kernel<<<grid, kAppendThreads, 0, stream>>>(
      static_cast<const uint4*>(k), k_stride / 8, static_cast<const uint4*>(v), v_stride / 8,
      slot_mapping, num_tokens, static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
      num_slots, row_elems / 16, k_inv, v_inv);
  return cudaGetLastError();
}

}  // namespace pkv

// ---------------------------------------------------------------------------
// Block copy for copy-on-write: for each (src, dst) pair, block dst of the K
// pool and of the V pool becomes a byte copy of block src.  One CTA copies
// one block of one pool (a contiguous run of block_size * row bytes) with
// 16-byte vectors, four in flight per thread; the grid strides over the
// 2 * num_pairs (pair, pool) items.  Pure HBM copy.
// ---------------------------------------------------------------------------
namespace pkv {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;

__global__ void __launch_bounds__(kCopyThreads)
copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                   const int32_t* __restrict__ pairs, int num_pairs, int num_blocks,
                   int64_t block_vec) {
  for (int item = blockIdx.x; item < 2 * num_pairs; item += gridDim.x) {
    const int p = item >> 1;
    const int32_t src = __ldg(pairs + 2 * p), dst = __ldg(pairs + 2 * p + 1);
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      if (threadIdx.x == 0 && (item & 1) == 0) atomicOr(&g_append_error, kErrBadBlockId);
      continue;
    }
    uint4* pool = (item & 1) ? v_cache : k_cache;
    const uint4* from = pool + int64_t(src) * block_vec;
    uint4* to = pool + int64_t(dst) * block_vec;
    for (int64_t base = 0; base < block_vec; base += int64_t(kCopyThreads) * kCopyUnroll) {
      uint4 r[kCopyUnroll];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const int64_t i = base + int64_t(u) * kCopyThreads + threadIdx.x;
        if (i < block_vec) r[u] = from[i];
      }
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const int64_t i = base + int64_t(u) * kCopyThreads + threadIdx.x;
        if (i < block_vec) to[i] = r[u];
      }
    }
  }
}

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs,
                               int num_blocks, int64_t block_bytes, cudaStream_t stream,
                               int num_sms) {
  const int64_t items = 2 * int64_t(num_pairs);
  const int64_t max_blocks = int64_t(num_sms) * 8;
  const int grid = int(items < max_blocks ? items : max_blocks);
  copy_blocks_kernel<<<grid, kCopyThreads, 0, stream>>>(
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), pairs, num_pairs, num_blocks,
      block_bytes / 16);
  return cudaGetLastError();
}

}  // namespace pkv

// ---------------------------------------------------------------------------
// FP8 pages -> bf16 pages for the chunked prefill over an FP8 cache.  Page j
// of sequence s (j < ceil(context_len / 16)) is widened into block
// s * max_blocks + j of a bf16 scratch pool, and entry (s, j) of a scratch
// block table names it.  e4m3 -> f16 -> f32 -> bf16 is exact: every e4m3
// value (3 mantissa bits, exponents 2^-9 .. 2^8) is a bf16 value.  One CTA
// widens one page of K and V; each thread moves 16 codes per step (one
// 16-byte load, two 16-byte stores per pool).
// ---------------------------------------------------------------------------
#include <cuda_fp16.h>

namespace pkv {

constexpr int kPageTokens = 16;

// Two floats -> packed f16x2 (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t pack_f16x2_cvt(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint16_t two) {
  uint32_t h2;
  asm("{\n\t.reg .b16 c;\n\tmov.b16 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}"
      : "=r"(h2)
      : "h"(two));
  const __half2 h = *reinterpret_cast<const __half2*>(&h2);
  const float2 f = __half22float2(h);
  return pack_bf16x2(f.x, f.y);
}

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two) {
  uint32_t h2;
  asm("{\n\t.reg .b16 c;\n\tmov.b16 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}"
      : "=r"(h2)
      : "h"(two));
  return h2;
}

__device__ __forceinline__ uint4 widen8_f16(uint32_t a, uint32_t b) {
  return make_uint4(e4m3x2_to_f16x2(uint16_t(a & 0xffffu)), e4m3x2_to_f16x2(uint16_t(a >> 16)),
                    e4m3x2_to_f16x2(uint16_t(b & 0xffffu)), e4m3x2_to_f16x2(uint16_t(b >> 16)));
}

__device__ __forceinline__ uint4 widen8(uint32_t a, uint32_t b) {
  return make_uint4(e4m3x2_to_bf16x2(uint16_t(a & 0xffffu)), e4m3x2_to_bf16x2(uint16_t(a >> 16)),
                    e4m3x2_to_bf16x2(uint16_t(b & 0xffffu)), e4m3x2_to_bf16x2(uint16_t(b >> 16)));
}

// order[r] = the sequence of rank r when sequences are sorted by context
// length, longest first, ties by index.  Every sequence's rank is the number
// of sequences before it in that order, so the ranks are a permutation of
// 0 .. num_seqs-1 whatever the lengths; the grid shares the num_seqs^2
// comparisons.
__device__ __forceinline__ void rank_by_length(const int32_t* __restrict__ lens, int num_seqs,
                                               int32_t* __restrict__ order) {
  const int stride = int(gridDim.x) * int(blockDim.x);
  for (int s = int(blockIdx.x) * int(blockDim.x) + int(threadIdx.x); s < num_seqs; s += stride) {
    const int key = __ldg(lens + s);
    int rank = 0;
    for (int t = 0; t < num_seqs; ++t) {
      const int other = __ldg(lens + t);
      rank += (other > key) || (other == key && t < s);
    }
    order[rank] = s;
  }
}

__global__ void __launch_bounds__(kAppendThreads)
widen_fp8_pages_kernel(const uint4* __restrict__ k8, const uint4* __restrict__ v8,
                       const int32_t* __restrict__ tables, const int32_t* __restrict__ lens,
                       int num_seqs, int max_blocks, int num_blocks, int page_vec16,
                       uint4* __restrict__ kdst, uint4* __restrict__ vdst,
                       int32_t* __restrict__ table_out, bool v_f16,
                       int32_t* __restrict__ seq_order) {
  if (seq_order) rank_by_length(lens, num_seqs, seq_order);
  const int64_t items = int64_t(num_seqs) * max_blocks;
  for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
    const int s = int(item / max_blocks), j = int(item - int64_t(s) * max_blocks);
    if (threadIdx.x == 0) table_out[item] = int32_t(item);
    const int len = min(max(__ldg(lens + s), 0), max_blocks * kPageTokens);
    if (j * kPageTokens >= len) continue;
    const int32_t src = __ldg(tables + item);
    const bool ok = src >= 0 && src < num_blocks;
    if (!ok && threadIdx.x == 0) atomicOr(&g_append_error, kErrBadBlockId);
    const uint4* ks = k8 + int64_t(ok ? src : 0) * page_vec16;
    const uint4* vs = v8 + int64_t(ok ? src : 0) * page_vec16;
    uint4* kd = kdst + item * page_vec16 * 2;  // 16 codes -> 32 bytes of bf16
    uint4* vd = vdst + item * page_vec16 * 2;
    for (int i = threadIdx.x; i < page_vec16; i += kAppendThreads) {
      const uint4 kc = ok ? __ldg(ks + i) : make_uint4(0, 0, 0, 0);
      const uint4 vc = ok ? __ldg(vs + i) : make_uint4(0, 0, 0, 0);
      kd[2 * i] = widen8(kc.x, kc.y);
      kd[2 * i + 1] = widen8(kc.z, kc.w);
      vd[2 * i] = v_f16 ? widen8_f16(vc.x, vc.y) : widen8(vc.x, vc.y);
      vd[2 * i + 1] = v_f16 ? widen8_f16(vc.z, vc.w) : widen8(vc.z, vc.w);
    }
  }
}

cudaError_t launch_widen_fp8_pages(const void* k8, const void* v8, const int32_t* tables,
                                   const int32_t* lens, int num_seqs, int max_blocks,
                                   int num_blocks, int64_t page_codes, void* kdst, void* vdst,
                                   int32_t* table_out, bool v_f16, int32_t* seq_order,
                                   cudaStream_t stream, int num_sms) {
  const int64_t items = int64_t(num_seqs) * max_blocks;
  const int64_t max_grid = int64_t(num_sms) * 8;
  const int grid = int(items < max_grid ? items : max_grid);
  widen_fp8_pages_kernel<<<grid, kAppendThreads, 0, stream>>>(
      static_cast<const uint4*>(k8), static_cast<const uint4*>(v8), tables, lens, num_seqs,
      max_blocks, num_blocks, int(page_codes / 16), static_cast<uint4*>(kdst),
      static_cast<uint4*>(vdst), table_out, v_f16, seq_order);
  return cudaGetLastError();
}

// bf16 V pages -> f16 pages for the prefill's single-product P V: page j of
// sequence s (j < ceil(context_len / 16)) into block s * max_blocks + j of an
// f16 scratch pool, named by entry (s, j) of a scratch table.  Exact for
// |v| in [2^-14, 65504]; smaller values become f16 subnormals (absolute error
// below 2^-25); a value of magnitude 65520 or more overflows and sets the f16
// range bit of the error word.
constexpr unsigned kErrFp16RangeAppend = 1u << 6;

__global__ void __launch_bounds__(kAppendThreads)
v_pages_to_f16_kernel(const uint4* __restrict__ v, const int32_t* __restrict__ tables,
                      const int32_t* __restrict__ lens, int num_seqs, int max_blocks,
                      int num_blocks, int page_vec, uint4* __restrict__ vdst,
                      int32_t* __restrict__ table_out, int32_t* __restrict__ seq_order) {
  if (seq_order) rank_by_length(lens, num_seqs, seq_order);
  const int64_t items = int64_t(num_seqs) * max_blocks;
  for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
    const int s = int(item / max_blocks), j = int(item - int64_t(s) * max_blocks);
    if (threadIdx.x == 0) table_out[item] = int32_t(item);
    const int len = min(max(__ldg(lens + s), 0), max_blocks * kPageTokens);
    if (j * kPageTokens >= len) continue;
    const int32_t src = __ldg(tables + item);
    const bool ok = src >= 0 && src < num_blocks;
    if (!ok && threadIdx.x == 0) atomicOr(&g_append_error, kErrBadBlockId);
    const uint4* vs = v + int64_t(ok ? src : 0) * page_vec;
    uint4* vd = vdst + item * page_vec;
    bool in_range = true;
    for (int i = threadIdx.x; i < page_vec; i += kAppendThreads) {
      const uint4 x = ok ? __ldg(vs + i) : make_uint4(0, 0, 0, 0);
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
      uint32_t o[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float a = bf16_lo_to_f32(w[c]), b = bf16_hi_to_f32(w[c]);
        in_range &= !(fabsf(a) >= 65520.f) && !(fabsf(b) >= 65520.f);
        o[c] = pack_f16x2_cvt(a, b);
      }
      vd[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (!in_range) atomicOr(&g_append_error, kErrFp16RangeAppend);
  }
}

cudaError_t launch_v_pages_to_f16(const void* v, const int32_t* tables, const int32_t* lens,
                                  int num_seqs, int max_blocks, int num_blocks, int64_t page_elems,
                                  void* vdst, int32_t* table_out, int32_t* seq_order,
                                  cudaStream_t stream, int num_sms) {
  const int64_t items = int64_t(num_seqs) * max_blocks;
  const int64_t max_grid = int64_t(num_sms) * 8;
  const int grid = int(items < max_grid ? items : max_grid);
  v_pages_to_f16_kernel<<<grid, kAppendThreads, 0, stream>>>(
      static_cast<const uint4*>(v), tables, lens, num_seqs, max_blocks, num_blocks,
      int(page_elems / 8), static_cast<uint4*>(vdst), table_out, seq_order);
  return cudaGetLastError();
}

}  // namespace pkv
