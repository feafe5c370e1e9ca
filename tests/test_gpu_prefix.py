"""Shared-prefix (cascade) decode: the prefix attended once for all
sequences on the tensor cores, the private pages by split-K, merged by
log-sum-exp -- equal to the plain paged decode and to the oracle."""

import pytest
import torch

from paged_kv_cache_52_gb300 import workloads as wl
from parity import DecodeStepOracle, assert_attention_close

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_52_gb300 import pagedkv
    pagedkv.get_device_error(clear=True)
    return pagedkv


def _decodes(m):
    P = m.q_prefill.shape[0]
    return wl.DecodeWorkload("shared-prefix decodes", m.q_decode, m.k_cache, m.v_cache,
                             m.k_new[P:], m.v_new[P:], m.slot_mapping[P:], m.decode_tables,
                             m.decode_lens, m.scale, {"lens": m.meta["decode_lens"]})


def _run(pk, w, prefix_blocks):
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    pk.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    mcl = max(w.meta["lens"])
    casc = pk.paged_decode_attention_shared_prefix(w.q, kc, vc, w.block_tables, w.context_lens,
                                                   w.scale, prefix_blocks, mcl)
    plain = pk.paged_decode_attention(w.q, kc, vc, w.block_tables, w.context_lens, w.scale,
                                      max_context_len=mcl)
    torch.cuda.synchronize()
    return casc, plain


@pytest.mark.parametrize("prefix,ndec,cap", [(64, 40, 600), (16, 7, 100), (1024, 30, 3000)])
def test_shared_prefix_matches_oracle_and_plain_decode(pk, prefix, ndec, cap):
    m = wl.make_mixed_workload(num_prefill=0, num_decode=ndec, shared_prefix=prefix,
                               decode_cap=cap)
    w = _decodes(m)
    ref = DecodeStepOracle(w, range(ndec)).output()
    for n in ("q", "k_cache", "v_cache", "k_new", "v_new", "slot_mapping", "block_tables",
              "context_lens"):
        setattr(w, n, getattr(w, n).to(DEV))
    casc, plain = _run(pk, w, prefix // 16)
    assert_attention_close(casc.cpu().numpy(), ref, f"cascade prefix {prefix}")
    assert_attention_close(casc.cpu().numpy(), plain.cpu().numpy(), "cascade vs plain")
    assert pk.get_device_error() == 0


def test_shared_prefix_full_mixed_step_decodes(pk):
    m = wl.make_mixed_workload(device=DEV, gen_device=DEV)
    w = _decodes(m)
    seqs = [0, 123, 247]
    ref = DecodeStepOracle(w, seqs).output()
    casc, plain = _run(pk, w, m.meta["shared_prefix"] // 16)
    assert_attention_close(casc[seqs].cpu().numpy(), ref, "cascade full")
    assert_attention_close(casc.cpu().numpy(), plain.cpu().numpy(), "cascade vs plain full")
    assert pk.get_device_error() == 0


def test_context_shorter_than_prefix_is_flagged(pk):
    m = wl.make_mixed_workload(num_prefill=0, num_decode=4, shared_prefix=64, decode_cap=300)
    w = _decodes(m)
    for n in ("q", "k_cache", "v_cache", "block_tables", "context_lens"):
        setattr(w, n, getattr(w, n).to(DEV))
    lens = w.context_lens.clone()
    lens[2] = 30                      # inside the 64-token prefix
    pk.get_device_error(clear=True)
    pk.paged_decode_attention_shared_prefix(w.q, w.k_cache, w.v_cache, w.block_tables, lens,
                                            w.scale, 4, int(lens.max()))
    assert pk.get_device_error(clear=True) & 0x4
