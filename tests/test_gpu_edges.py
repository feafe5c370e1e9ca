"""Boundary cases of the GPU path against the oracle: partitions at the
largest size the kernels stage (1024 pages), contexts that exactly fill the
block table, single-token and tile-multiple chunks that cover the whole
context, and every decode-family kernel on the same boundary workload."""

import numpy as np
import pytest
import torch

from paged_kv_cache_52_gb300 import workloads as wl
from parity import DecodeStepOracle, PrefillStepOracle, assert_attention_close

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_52_gb300 import pagedkv
    pagedkv.get_device_error(clear=True)
    return pagedkv


def _to_dev(w, names):
    for n in names:
        setattr(w, n, getattr(w, n).to(DEV))
    return w


DEC = ("q", "k_cache", "v_cache", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens")
# 16384 tokens = exactly 1024 pages (one full partition at the largest size),
# 20000 = 1250 pages (a full partition and a ragged one), 16385 = one past it
BIG_LENS = [16384, 20000, 16385, 1]


def _big_decode_workload(hq=8, hkv=2, d=64):
    spec = wl.DecodeSpec("edges", 12, len(BIG_LENS), hq, hkv, d, lens=tuple(BIG_LENS))
    return wl.make_decode_workload(spec, lens_override=BIG_LENS)


@pytest.mark.parametrize("pb", [1024, 1000, 0])
def test_decode_at_the_largest_partition(pk, pb):
    w = _big_decode_workload()
    ref = DecodeStepOracle(w, range(len(BIG_LENS))).output()
    w = _to_dev(w, DEC)
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    pk.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    out = pk.paged_decode_attention(w.q, kc, vc, w.block_tables, w.context_lens, w.scale,
                                    max_context_len=max(BIG_LENS), partition_blocks=pb)
    torch.cuda.synchronize()
    assert_attention_close(out.cpu().numpy(), ref, f"decode pb={pb}")
    assert pk.get_device_error(clear=True) == 0


def test_fp8_decode_at_the_largest_partition(pk):
    from test_gpu_fp8 import _fp8_oracle
    w = _to_dev(_big_decode_workload(16, 2, 128), DEC)
    kc8, vc8 = wl.fp8_pools(w, 0.03125, 0.03125)
    ref = _fp8_oracle(w, kc8, vc8, 0.03125, 0.03125, range(len(BIG_LENS)))
    kc, vc = kc8.clone(), vc8.clone()
    pk.kv_append_fp8(w.k_new, w.v_new, w.slot_mapping, kc, vc, 0.03125, 0.03125)
    out = pk.paged_decode_attention_fp8(w.q, kc, vc, w.block_tables, w.context_lens, w.scale,
                                        0.03125, 0.03125, max_context_len=max(BIG_LENS),
                                        partition_blocks=1024)
    torch.cuda.synchronize()
    assert_attention_close(out.cpu().numpy(), ref, "fp8 decode pb=1024")
    assert pk.get_device_error(clear=True) == 0


def test_context_exactly_filling_the_block_table(pk):
    # tables exactly as wide as the longest sequence needs: 16 * width tokens
    lens = [16 * 7, 16 * 7 - 1, 5]
    spec = wl.DecodeSpec("full table", 13, len(lens), 8, 4, 128, lens=tuple(lens))
    w = wl.make_decode_workload(spec, lens_override=lens)
    w.block_tables = w.block_tables[:, :7].contiguous()
    ref = DecodeStepOracle(w, range(len(lens))).output()
    w = _to_dev(w, DEC)
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    pk.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    for pb in (0, 1, 7):
        out = pk.paged_decode_attention(w.q, kc, vc, w.block_tables, w.context_lens, w.scale,
                                        max_context_len=max(lens), partition_blocks=pb)
        torch.cuda.synchronize()
        assert_attention_close(out.cpu().numpy(), ref, f"full table pb={pb}")
    assert pk.get_device_error(clear=True) == 0


PF = ("k_cache", "v_cache", "k_new", "v_new", "slot_mapping", "q_prefill", "q_start",
      "prefill_tables", "prefill_lens")


@pytest.mark.parametrize("causal", [True, False])
def test_prefill_chunks_covering_the_whole_context(pk, causal):
    # prior 0: the chunk is the whole context -- 1 token, a 16-token page, a
    # 128-key tile, 256 (two query tiles of one CTA at G = 8), 257
    chunks = [1, 16, 128, 256, 257]
    w = wl.make_chunked_workload(64, 8, 128, [0] * len(chunks), chunks)
    ref = PrefillStepOracle(w, range(len(chunks)), causal=causal).output()
    w = _to_dev(w, PF)
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    pk.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    out = pk.paged_prefill_attention(w.q_prefill, w.q_start, kc, vc, w.prefill_tables,
                                     w.prefill_lens, causal, w.scale, max_q_len=max(chunks))
    torch.cuda.synchronize()
    assert_attention_close(out.cpu().numpy(), ref, f"whole-context chunks causal={causal}")
    assert pk.get_device_error(clear=True) == 0


def test_verify_at_the_largest_partition(pk):
    K = 2
    lens = [16384, 20000, 17]
    w = wl.make_chunked_workload(16, 2, 64, [L - K for L in lens], [K] * len(lens),
                                 config_id=14)
    ref = PrefillStepOracle(w, range(len(lens)), causal=True).output()
    w = _to_dev(w, PF)
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    pk.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    q = w.q_prefill.view(len(lens), K, 16, 64)
    out = pk.paged_verify_attention(q, kc, vc, w.prefill_tables, w.prefill_lens, w.scale,
                                    max_context_len=max(lens), partition_blocks=1024)
    torch.cuda.synchronize()
    assert_attention_close(out.view(-1, 16, 64).cpu().numpy(), ref, "verify pb=1024")
    assert pk.get_device_error(clear=True) == 0
