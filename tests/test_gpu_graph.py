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


def test_mixed_step_captured_in_one_graph(pk):
    """append + chunked prefill + decode captured once and replayed: same
    results as the eager calls, and the prefill rows match the oracle."""
    from parity import PrefillStepOracle
    m = wl.make_mixed_workload(num_prefill=3, num_decode=9, chunk=100, prior_range=(0, 400),
                               shared_prefix=32, decode_cap=900)
    pref = PrefillStepOracle(m, range(3)).output()
    for n in ("k_cache", "v_cache", "k_new", "v_new", "slot_mapping", "q_prefill", "q_start",
              "prefill_tables", "prefill_lens", "q_decode", "decode_tables", "decode_lens"):
        setattr(m, n, getattr(m, n).to(DEV))
    kc, vc = m.k_cache.clone(), m.v_cache.clone()
    pout = torch.empty(m.q_prefill.shape, dtype=torch.float32, device=DEV)
    dout = torch.empty(m.q_decode.shape, dtype=torch.float32, device=DEV)
    mdl = max(m.meta["decode_lens"])
    ws = pk.decode_workspace(m.q_decode.shape[0], m.q_decode.shape[1], kc.shape[2], kc.shape[3],
                             mdl, DEV)

    def step():
        pk.kv_append(m.k_new, m.v_new, m.slot_mapping, kc, vc)
        pk.paged_prefill_attention(m.q_prefill, m.q_start, kc, vc, m.prefill_tables,
                                   m.prefill_lens, True, m.scale, out=pout, max_q_len=100)
        pk.paged_decode_attention(m.q_decode, kc, vc, m.decode_tables, m.decode_lens, m.scale,
                                  out=dout, max_context_len=mdl, workspace=ws)

    step()                                    # eager (also sets kernel attributes)
    torch.cuda.synchronize()
    eager_p, eager_d = pout.clone(), dout.clone()
    pout.zero_(), dout.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(pout, eager_p) and torch.equal(dout, eager_d)
    assert_attention_close(pout.cpu().numpy(), pref, "graph mixed step prefill")
    assert pk.get_device_error() == 0
