"""Decode replayed from CUDA graphs captured per batch-size bucket (padded
sequences have context_len 0 and slot -1) matches the oracle."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_52_gb300 import workloads as wl
from parity import DecodeStepOracle, assert_attention_close

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_52_gb300 import pagedkv
    pagedkv.get_device_error(clear=True)
    return pagedkv


def _dev(w):
    for n in ("q", "k_cache", "v_cache", "k_new", "v_new", "slot_mapping", "block_tables",
              "context_lens"):
        setattr(w, n, getattr(w, n).to(DEV))
    return w


def test_bucketed_graph_replay_matches_oracle(pk):
    from paged_kv_cache_52_gb300.graphs import DecodeGraphRunner
    lens = [1500, 37, 4096, 800, 2222, 16, 17, 3000, 1, 640, 999]
    w = wl.make_decode_workload(wl.GQA_70B, lens_override=lens)
    ref_all = DecodeStepOracle(w, range(len(lens)))
    ref = ref_all.output()
    w = _dev(w)
    kc0 = wl.bf16_bits(w.k_cache)
    runner = DecodeGraphRunner(w.k_cache, w.v_cache, w.q_heads, w.block_tables.shape[1],
                               max(lens), w.scale, buckets=(4, 16))
    # batch of 11 -> bucket 16 (5 padded rows)
    out = runner.run(w.q, w.k_new, w.v_new, w.slot_mapping, w.block_tables,
                     w.context_lens).clone()
    torch.cuda.synchronize()
    assert_attention_close(out.cpu().numpy(), ref, "graph bucket 16")
    assert runner.buckets[16].graph is not None
    # the append went into the pools through the graph, bit-exact
    k_ref, _ = oracle.kv_append(wl.bf16_bits(w.k_new), wl.bf16_bits(w.v_new),
                                w.slot_mapping.cpu().numpy(), kc0, wl.bf16_bits(w.v_cache))
    assert np.array_equal(wl.bf16_bits(w.k_cache), k_ref)
    # replay again with a smaller live batch -> bucket 4
    sub = [2, 0, 7]
    out2 = runner.run(w.q[sub], w.k_new[sub], w.v_new[sub], w.slot_mapping[sub],
                      w.block_tables[sub], w.context_lens[sub])
    torch.cuda.synchronize()
    assert_attention_close(out2.cpu().numpy(), ref[sub], "graph bucket 4")
    # and the first bucket's graph replays unchanged
    out3 = runner.run(w.q, w.k_new, w.v_new, w.slot_mapping, w.block_tables, w.context_lens)
    torch.cuda.synchronize()
    assert torch.equal(out3, out)
    assert pk.get_device_error() == 0
    with pytest.raises(ValueError):
        runner.bucket_for(17)
