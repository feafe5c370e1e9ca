"""Multi-query decode (speculative verification) on the GPU against the CPU
oracle: K drafted tokens per sequence, already appended, each attending over
the context up to its own position -- the oracle's causal prefill of a
K-token chunk."""

import numpy as np
import pytest
import torch

from paged_kv_cache_52_gb300 import workloads as wl
from parity import PrefillStepOracle, assert_attention_close

pytestmark = pytest.mark.gpu

DEV = "cuda"
NAMES = ("k_cache", "v_cache", "k_new", "v_new", "slot_mapping", "q_prefill", "q_start",
         "prefill_tables", "prefill_lens")


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_52_gb300 import pagedkv
    pagedkv.get_device_error(clear=True)
    return pagedkv


def _workload(hq, hkv, d, lens, K, config_id=8, device="cpu"):
    return wl.make_chunked_workload(hq, hkv, d, [L - K for L in lens], [K] * len(lens),
                                    config_id=config_id, device=device, gen_device=device)


def _dev(w):
    for n in NAMES:
        setattr(w, n, getattr(w, n).to(DEV))
    return w


def _run(pk, w, K, pb=0, poison=False):
    S = w.prefill_lens.shape[0]
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    pk.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    if poison:  # rows past each length in its last page hold NaN
        tables = w.prefill_tables.cpu().numpy()
        for s, L in enumerate(w.prefill_lens.cpu().tolist()):
            if L % 16:
                b = int(tables[s, (L - 1) // 16])
                kc[b, L % 16:] = float("nan")
                vc[b, L % 16:] = float("nan")
    hq, d = w.q_prefill.shape[1], w.q_prefill.shape[2]
    q = w.q_prefill.view(S, K, hq, d)
    out = pk.paged_verify_attention(q, kc, vc, w.prefill_tables, w.prefill_lens, w.scale,
                                    max_context_len=int(w.prefill_lens.max()),
                                    partition_blocks=pb)
    torch.cuda.synchronize()
    return out.view(S * K, hq, d)


LENS = [4, 17, 33, 300, 1000, 16, 250, 129]


@pytest.mark.parametrize("hq,hkv,d,K", [(64, 8, 128, 1), (64, 8, 128, 2), (64, 8, 128, 4),
                                         (16, 4, 64, 4), (8, 8, 128, 16), (8, 8, 128, 3),
                                         (32, 2, 64, 2), (16, 16, 64, 32)])
@pytest.mark.parametrize("pb", [0, 2])
def test_verify_groups_tokens_and_ragged_lengths(pk, hq, hkv, d, K, pb):
    lens = [max(L, K) for L in LENS]
    w = _workload(hq, hkv, d, lens, K)
    ref = PrefillStepOracle(w, range(len(lens)), causal=True).output()
    out = _run(pk, _dev(w), K, pb)
    assert_attention_close(out.cpu().numpy(), ref, f"verify {hq}/{hkv} d{d} K={K} pb={pb}")
    assert pk.get_device_error(clear=True) == 0


@pytest.mark.parametrize("K", [2, 4])
def test_verify_nan_rows_past_the_length(pk, K):
    lens = [max(L, K) for L in LENS]
    w = _workload(64, 8, 128, lens, K)
    ref = PrefillStepOracle(w, range(len(lens)), causal=True).output()
    out = _run(pk, _dev(w), K, 2, poison=True)
    assert_attention_close(out.cpu().numpy(), ref, f"verify NaN tails K={K}")
    assert pk.get_device_error(clear=True) == 0


def test_verify_full_size_70b_gqa_whole_batch(pk):
    # 256 sequences, contexts U[1024, 8192] after appending 4 drafted tokens,
    # 0.1% of K rows x100; every query row of every sequence against the
    # oracle's causal prefill of 4-token chunks
    K = 4
    g = torch.Generator().manual_seed(1000 * 3 + 5)
    lens = torch.randint(1024, 8193, (256,), generator=g).tolist()
    w = _workload(64, 8, 128, lens, K, config_id=9, device=DEV)
    flat = w.k_cache.view(-1, 128)
    rows = torch.randperm(flat.shape[0], generator=torch.Generator().manual_seed(3007))
    rows = rows[:round(0.001 * flat.shape[0])].to(DEV)
    flat[rows] = (flat[rows].float() * 100).to(torch.bfloat16)
    orc = PrefillStepOracle(w, range(256), causal=True)
    ref = orc.output()
    out = _run(pk, _dev(w), K)
    assert_attention_close(out.cpu().numpy(), ref, "verify 70B-GQA K=4")
    assert torch.isfinite(out).all()
    assert pk.get_device_error(clear=True) == 0


def test_verify_context_shorter_than_the_drafts_is_flagged(pk):
    K = 4
    w = _dev(_workload(8, 2, 64, [4, 20], K))
    lens = w.prefill_lens.clone()
    lens[0] = 2                                  # tokens 0 and 1 would sit before position 0
    S = 2
    q = w.q_prefill.view(S, K, 8, 64)
    pk.get_device_error(clear=True)
    out = pk.paged_verify_attention(q, w.k_cache, w.v_cache, w.prefill_tables, lens, w.scale,
                                    max_context_len=20)
    torch.cuda.synchronize()
    assert pk.get_device_error(clear=True) & 0x10
    assert torch.isfinite(out).all()
    assert (out[0, :2] == 0).all()               # no key for tokens before position 0


def test_verify_repeatable_bitwise(pk):
    w = _dev(_workload(64, 8, 128, [900, 2500, 64], 4))
    a = _run(pk, w, 4)
    b = _run(pk, w, 4)
    assert torch.equal(a, b)
