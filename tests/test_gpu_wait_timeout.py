"""Failure detection on the GPU without a fault: the bounded mbarrier wait
every kernel uses is made to run out on a barrier phase that nothing
completes.  The timeout bit must reach the host, the wait must last longer
with a larger poll limit (the bound is what ends it), and the context must
stay usable: a decode step afterwards still matches the oracle."""

import pytest
import torch

from paged_kv_cache_52_gb300 import workloads as wl
from parity import DecodeStepOracle, assert_attention_close

pytestmark = pytest.mark.gpu

DEV = "cuda"
WAIT_TIMEOUT = 0x8


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_52_gb300 import pagedkv
    pagedkv.get_device_error(clear=True)
    return pagedkv


def test_bounded_wait_runs_out_and_the_context_stays_usable(pk):
    short = pk.wait_timeout_probe(1 << 10)
    assert pk.get_device_error(clear=True) == WAIT_TIMEOUT
    long_ = pk.wait_timeout_probe(1 << 14)
    assert pk.get_device_error(clear=True) == WAIT_TIMEOUT
    assert 0 < short < long_
    # the same timeout through the stream-ordered query: PKV_ETIMEOUT
    pk.wait_timeout_probe(1 << 10)
    status, bits = pk.get_last_device_error()
    assert status == pk.PKV_ETIMEOUT and bits == WAIT_TIMEOUT
    assert pk.get_last_device_error() == (0, 0)
    # the context is intact after the timeouts
    w = wl.make_decode_workload(wl.TINY)
    ref = DecodeStepOracle(w, range(w.num_seqs)).output()
    kc, vc = w.k_cache.to(DEV), w.v_cache.to(DEV)
    pk.kv_append(w.k_new.to(DEV), w.v_new.to(DEV), w.slot_mapping.to(DEV), kc, vc)
    out = pk.paged_decode_attention(w.q.to(DEV), kc, vc, w.block_tables.to(DEV),
                                    w.context_lens.to(DEV), w.scale,
                                    max_context_len=max(w.meta["lens"]), partition_blocks=2)
    torch.cuda.synchronize()
    assert_attention_close(out.cpu().numpy(), ref, "decode after the probe")
    assert pk.get_device_error(clear=True) == 0
