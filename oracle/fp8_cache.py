"""Oracle for an FP8 (e4m3) paged KV cache with per-tensor scales.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The pages name FP8 KV caches as the next step in shrinking KV bytes ("Cache
KV, attention et optimisation de l'inference", section "Utilisez-le": vLLM
served with ``--kv-cache-dtype fp8``; "第 10 讲：推理（Inference）": fewer bits,
fewer bytes, faster memory-bound decode) but fix no format.  Reading taken:

* element format e4m3 ("fn": 1 sign, 4 exponent bits with bias 7, 3 mantissa
  bits, no infinities, S.1111.111 is NaN, largest finite 448);
* one float32 scale per pool (``k_scale``, ``v_scale``): a cached value
  stands for ``e4m3 * scale``;
* appending quantizes ``q = e4m3(float32(x) * inv_scale)`` with
  ``inv_scale = float32(1) / float32(scale)``, rounding to nearest even and
  saturating finite overflow to +-448 ("satfinite");
* attention over an FP8 cache is the float64 attention of the dequantized
  cache.
"""

from __future__ import annotations

import numpy as np

from .paged_attention import _as_f64, kv_append, paged_decode_attention, paged_prefill_attention

E4M3_MAX = 448.0
E4M3_NAN = 0x7F


def e4m3_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of e4m3 bit patterns (uint8): subnormals m * 2^-9, normals
    (1 + m/8) * 2^(e - 7), S.1111.111 = NaN."""
    b = np.asarray(bits).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 0x7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


def _round_half_even(q: np.ndarray) -> np.ndarray:
    m = np.floor(q)
    r = q - m
    odd = np.mod(m, 2.0) == 1.0
    return np.where((r > 0.5) | ((r == 0.5) & odd), m + 1.0, m)


def f32_to_e4m3_bits(x) -> np.ndarray:
    """Round float32 values to e4m3 (nearest, ties to even mantissa), finite
    overflow and infinities saturating to +-448, NaN to the NaN pattern.

    Subnormal range (|x| < 2^-6): the code is round(|x| / 2^-9); a result of 8
    is exactly the smallest normal.  Normal range: with 2^e <= |x| < 2^(e+1),
    the mantissa code is round((|x| / 2^e - 1) * 8), carrying into the
    exponent when it reaches 8."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)  # exact widening
    a = np.abs(x)
    sign = np.where(np.signbit(x), 0x80, 0).astype(np.int64)
    with np.errstate(divide="ignore", invalid="ignore"):
        # subnormal candidates
        sub = _round_half_even(a / 2.0 ** -9)
        # normal candidates: exact binade via frexp (a = f * 2^k, 0.5 <= f < 1)
        f, k = np.frexp(np.where(a > 0, a, 1.0))
        e = k.astype(np.int64) - 1
        mant = _round_half_even((a / np.exp2(e.astype(np.float64)) - 1.0) * 8.0)
        carry = mant >= 8.0
        e = np.where(carry, e + 1, e)
        mant = np.where(carry, 0.0, mant)
        field = e + 7
        normal_code = (field << 3) | mant.astype(np.int64)
        overflow = (field > 15) | ((field == 15) & (mant == 7.0))
        code = np.where(a < 2.0 ** -6, sub.astype(np.int64), normal_code)
        code = np.where(overflow | (a >= E4M3_MAX), 0x7E, code)
    code = code | sign
    code = np.where(np.isnan(x), E4M3_NAN, code)
    return code.astype(np.uint8)


def quantize_rows(rows, scale) -> np.ndarray:
    """e4m3 codes of ``float32(rows) * (float32(1) / float32(scale))``."""
    inv = np.float32(1.0) / np.float32(scale)
    return f32_to_e4m3_bits(_as_f64(rows).astype(np.float32) * inv)


def kv_append_fp8(k_new, v_new, slot_mapping, k_cache_bits, v_cache_bits, k_scale, v_scale):
    """Quantize the new K/V rows and scatter them (slot -1 skips)."""
    return kv_append(quantize_rows(k_new, k_scale), quantize_rows(v_new, v_scale),
                     slot_mapping, k_cache_bits, v_cache_bits)


# e4m3_bits_to_f64 evaluated once for each of the 256 codes: dequantizing a
# pool then indexes this table, which gives the same values as applying the
# function element by element, at a fraction of the cost on large pools.
_E4M3_VALUES = e4m3_bits_to_f64(np.arange(256, dtype=np.uint8))


def dequantize(cache_bits, scale) -> np.ndarray:
    bits = np.asarray(cache_bits)
    if bits.dtype != np.uint8:
        raise TypeError(f"expected uint8 e4m3 codes, got {bits.dtype}")
    return _E4M3_VALUES[bits] * float(np.float32(scale))


def paged_decode_attention_fp8(q, k_cache_bits, v_cache_bits, block_tables, context_lens,
                               scale, k_scale, v_scale):
    """Decode attention over the dequantized FP8 pools."""
    return paged_decode_attention(q, dequantize(k_cache_bits, k_scale),
                                  dequantize(v_cache_bits, v_scale), block_tables,
                                  context_lens, scale)


def paged_prefill_attention_fp8(q, q_start, k_cache_bits, v_cache_bits, block_tables,
                                context_lens, causal, scale, k_scale, v_scale):
    """Chunked prefill attention over the dequantized FP8 pools."""
    return paged_prefill_attention(q, q_start, dequantize(k_cache_bits, k_scale),
                                   dequantize(v_cache_bits, v_scale), block_tables,
                                   context_lens, causal, scale)
