"""Pins of the FP8 (e4m3) cache oracle: the format against torch's own
float8_e4m3fn conversion and closed forms, and FP8 decode against the pinned
bf16 oracle on the dequantized values."""

import numpy as np
import torch

import oracle
from paged_kv_cache_52_gb300 import workloads as wl


def test_e4m3_decode_matches_torch_for_all_256_codes():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_bits_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert np.array_equal(mine[~np.isnan(mine)], ref[~np.isnan(ref)])


def test_e4m3_encode_matches_torch_in_range():
    g = torch.Generator().manual_seed(4)
    x = torch.randn(20000, generator=g) * torch.exp(torch.randn(20000, generator=g) * 3)
    x = x[x.abs() < 460]
    # every code's value, and every midpoint between neighbouring codes (ties)
    vals = oracle.e4m3_bits_to_f64(np.arange(0, 0x7F, dtype=np.uint8))
    mids = (vals[1:] + vals[:-1]) / 2
    extra = torch.tensor(np.concatenate([vals, mids, -vals, -mids]), dtype=torch.float32)
    x = torch.cat([x, extra])
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = oracle.f32_to_e4m3_bits(x.numpy())
    assert np.array_equal(mine, ref)


def test_e4m3_saturation_closed_forms():
    enc = oracle.f32_to_e4m3_bits
    assert enc([448.0])[0] == 0x7E and enc([463.9])[0] == 0x7E      # stays finite
    assert enc([464.0])[0] == 0x7E and enc([1e30])[0] == 0x7E      # satfinite, not NaN
    assert enc([np.inf])[0] == 0x7E and enc([-np.inf])[0] == 0xFE
    assert enc([np.nan])[0] == 0x7F
    assert enc([2.0 ** -10])[0] == 0x00                           # tie to even (zero)
    assert enc([3 * 2.0 ** -10])[0] == 0x02                       # tie to even (2 * 2^-9)
    assert oracle.e4m3_bits_to_f64(np.array([0x08], np.uint8))[0] == 2.0 ** -6


def test_fp8_decode_equals_bf16_decode_of_dequantized_cache():
    # with power-of-two scales every dequantized value is exactly a bf16 value
    w = wl.make_decode_workload(wl.TINY)
    k_scale, v_scale = 0.0625, 0.03125
    kc8 = oracle.quantize_rows(wl.bf16_bits(w.k_cache), k_scale)
    vc8 = oracle.quantize_rows(wl.bf16_bits(w.v_cache), v_scale)
    kc8, vc8 = oracle.kv_append_fp8(wl.bf16_bits(w.k_new), wl.bf16_bits(w.v_new),
                                    w.slot_mapping.numpy(), kc8, vc8, k_scale, v_scale)
    got = oracle.paged_decode_attention_fp8(wl.bf16_bits(w.q), kc8, vc8, w.block_tables.numpy(),
                                            w.context_lens.numpy(), w.scale, k_scale, v_scale)
    kb = oracle.f64_to_bf16_bits(oracle.dequantize(kc8, k_scale))
    vb = oracle.f64_to_bf16_bits(oracle.dequantize(vc8, v_scale))
    assert np.array_equal(oracle.bf16_bits_to_f64(kb), oracle.dequantize(kc8, k_scale))
    ref = oracle.paged_decode_attention(wl.bf16_bits(w.q), kb, vb, w.block_tables.numpy(),
                                        w.context_lens.numpy(), w.scale)
    assert np.array_equal(got, ref)


def test_fp8_quantization_error_is_bounded():
    # e4m3 keeps 3 mantissa bits: relative error <= 2^-4 for normal values
    g = torch.Generator().manual_seed(9)
    x = (torch.randn(5000, generator=g) * 3).numpy().astype(np.float32)
    scale = np.float32(0.05)
    deq = oracle.dequantize(oracle.quantize_rows(x, scale), scale)
    inv = np.float32(1) / scale
    normal = np.abs(x * inv) >= 2.0 ** -6
    assert np.all(np.abs(deq - x)[normal] <= np.abs(x)[normal] * 2.0 ** -4 * 1.001)


def _fp8_chunked(k_scale, v_scale):
    w = wl.make_chunked_workload(8, 2, 64, [0, 40, 17], [5, 30, 1])
    kc8 = oracle.quantize_rows(wl.bf16_bits(w.k_cache), k_scale)
    vc8 = oracle.quantize_rows(wl.bf16_bits(w.v_cache), v_scale)
    kc8, vc8 = oracle.kv_append_fp8(wl.bf16_bits(w.k_new), wl.bf16_bits(w.v_new),
                                    w.slot_mapping.numpy(), kc8, vc8, k_scale, v_scale)
    return w, kc8, vc8


def test_fp8_prefill_equals_bf16_prefill_of_dequantized_cache():
    k_scale, v_scale = 0.0625, 0.03125
    w, kc8, vc8 = _fp8_chunked(k_scale, v_scale)
    args = (wl.bf16_bits(w.q_prefill), w.q_start.numpy())
    tail = (w.prefill_tables.numpy(), w.prefill_lens.numpy(), True, w.scale)
    got = oracle.paged_prefill_attention_fp8(*args, kc8, vc8, *tail, k_scale, v_scale)
    kb = oracle.f64_to_bf16_bits(oracle.dequantize(kc8, k_scale))
    vb = oracle.f64_to_bf16_bits(oracle.dequantize(vc8, v_scale))
    assert np.array_equal(got, oracle.paged_prefill_attention(*args, kb, vb, *tail))


def test_fp8_causal_prefill_equals_repeated_fp8_decode():
    k_scale, v_scale = 2.0, 0.03125
    w, kc8, vc8 = _fp8_chunked(k_scale, v_scale)
    q = wl.bf16_bits(w.q_prefill)
    qs = w.q_start.numpy()
    tables, lens = w.prefill_tables.numpy(), w.prefill_lens.numpy()
    got = oracle.paged_prefill_attention_fp8(q, qs, kc8, vc8, tables, lens, True, w.scale,
                                             k_scale, v_scale)
    for s in range(len(lens)):
        n = int(qs[s + 1] - qs[s])
        for i in range(n):
            row = int(qs[s]) + i
            ref = oracle.paged_decode_attention_fp8(q[row][None], kc8, vc8, tables[s:s + 1],
                                                    [int(lens[s]) - n + i + 1], w.scale,
                                                    k_scale, v_scale)
            np.testing.assert_allclose(got[row], ref[0], rtol=0, atol=1e-12)


def test_dequantize_table_equals_the_decoder():
    # the pool dequantizer indexes a table of the decoder's value for each
    # of the 256 codes: the same values, NaN for NaN, bit for bit
    codes = np.arange(256, dtype=np.uint8).reshape(16, 16)
    for scale in (1.0, 0.03125, 3.0):
        a = oracle.fp8_cache.e4m3_bits_to_f64(codes) * float(np.float32(scale))
        b = oracle.fp8_cache.dequantize(codes, scale)
        assert np.array_equal(a, b, equal_nan=True)
