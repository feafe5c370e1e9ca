"""Rows of a sequence's last page past its length may hold anything -- a pool
from torch.empty, a freed block's old content, or NaN.  Their attention
weight is zero, and the kernels must keep 0 * V exactly 0: with every such row
set to NaN (bf16) or to the e4m3 NaN code, decode (bf16 and FP8) and chunked
prefill still match the oracle, which never reads those rows."""

import numpy as np
import pytest
import torch

from paged_kv_cache_52_gb300 import workloads as wl
from parity import DecodeStepOracle, PrefillStepOracle, assert_attention_close

pytestmark = pytest.mark.gpu

DEV = "cuda"
LENS = [1, 15, 17, 33, 200, 161, 250, 3]


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_52_gb300 import pagedkv
    pagedkv.get_device_error(clear=True)
    return pagedkv


def poison_tail_rows(k_cache, v_cache, tables, lens, value):
    """Set the rows past each sequence's length in its last page to `value`."""
    tables = tables.cpu().numpy()
    for s, L in enumerate(int(x) for x in lens):
        if L % 16:
            b = int(tables[s, (L - 1) // 16])
            k_cache[b, L % 16:] = value
            v_cache[b, L % 16:] = value
    return k_cache, v_cache


def _dev(w, names):
    for n in names:
        setattr(w, n, getattr(w, n).to(DEV))
    return w


DECODE_NAMES = ("q", "k_cache", "v_cache", "k_new", "v_new", "slot_mapping", "block_tables",
                "context_lens")


@pytest.mark.parametrize("hq,hkv,d", [(8, 8, 128), (16, 4, 64), (64, 8, 128), (16, 1, 128)])
@pytest.mark.parametrize("pb", [0, 2])
def test_bf16_decode_ignores_nan_tail_rows(pk, hq, hkv, d, pb):
    spec = wl.DecodeSpec("tails", 14, len(LENS), hq, hkv, d, lens=tuple(LENS))
    w = wl.make_decode_workload(spec, lens_override=LENS)
    ref = DecodeStepOracle(w, range(w.num_seqs)).output()
    w = _dev(w, DECODE_NAMES)
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    pk.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    poison_tail_rows(kc, vc, w.block_tables, LENS, float("nan"))
    out = pk.paged_decode_attention(w.q, kc, vc, w.block_tables, w.context_lens, w.scale,
                                    max_context_len=max(LENS), partition_blocks=pb)
    torch.cuda.synchronize()
    assert_attention_close(out.cpu().numpy(), ref, f"bf16 decode {hq}/{hkv} d{d} pb={pb}")
    assert pk.get_device_error(clear=True) == 0


@pytest.mark.parametrize("hq,hkv", [(8, 8), (64, 8), (16, 16)])
@pytest.mark.parametrize("pb", [0, 3])
def test_fp8_decode_ignores_nan_tail_codes(pk, hq, hkv, pb):
    from test_gpu_fp8 import _fp8_oracle
    spec = wl.DecodeSpec("fp8 tails", 15, len(LENS), hq, hkv, 128, lens=tuple(LENS))
    w = _dev(wl.make_decode_workload(spec, lens_override=LENS), DECODE_NAMES)
    ks, vs = 0.03125, 0.03125
    kc8, vc8 = wl.fp8_pools(w, ks, vs)
    ref = _fp8_oracle(w, kc8, vc8, ks, vs, range(len(LENS)))
    kc, vc = kc8.clone(), vc8.clone()
    pk.kv_append_fp8(w.k_new, w.v_new, w.slot_mapping, kc, vc, ks, vs)
    poison_tail_rows(kc, vc, w.block_tables, LENS, 0x7F)          # e4m3 NaN
    out = pk.paged_decode_attention_fp8(w.q, kc, vc, w.block_tables, w.context_lens, w.scale,
                                        ks, vs, max_context_len=max(LENS), partition_blocks=pb)
    torch.cuda.synchronize()
    assert_attention_close(out.cpu().numpy(), ref, f"fp8 decode {hq}/{hkv} pb={pb}")
    assert pk.get_device_error(clear=True) == 0


PRIORS = [0, 40, 17, 300, 1000, 5, 3]
CHUNKS = [5, 130, 1, 129, 64, 16, 3]


@pytest.mark.parametrize("hq,hkv,d", [(8, 8, 128), (16, 4, 64), (64, 8, 128)])
@pytest.mark.parametrize("causal", [True, False])
def test_prefill_ignores_nan_tail_rows(pk, hq, hkv, d, causal):
    w = wl.make_chunked_workload(hq, hkv, d, PRIORS, CHUNKS)
    ref = PrefillStepOracle(w, range(len(CHUNKS)), causal=causal).output()
    w = _dev(w, ("k_cache", "v_cache", "k_new", "v_new", "slot_mapping", "q_prefill", "q_start",
                 "prefill_tables", "prefill_lens"))
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    pk.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    lens = w.prefill_lens.cpu().tolist()
    assert any(L % 16 for L in lens)
    poison_tail_rows(kc, vc, w.prefill_tables, lens, float("nan"))
    out = pk.paged_prefill_attention(w.q_prefill, w.q_start, kc, vc, w.prefill_tables,
                                     w.prefill_lens, causal, w.scale, max_q_len=max(CHUNKS))
    torch.cuda.synchronize()
    assert_attention_close(out.cpu().numpy(), ref, f"prefill {hq}/{hkv} d{d} causal={causal}")
    assert pk.get_device_error(clear=True) == 0
