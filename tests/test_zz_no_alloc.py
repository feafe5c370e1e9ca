"""The no-allocation decode entry point (for callers that may not call
cudaMalloc: fixed memory budgets, plug-ins handed device buffers, serving
loops that must not allocate mid-step) matches the regular entry point.

The file name sorts last so that a run stopping at the first failure has run
every other test first.  It also passes alone in a fresh process.
"""

import ctypes

import pytest
import torch

from paged_kv_cache_52_gb300 import workloads as wl
from parity import assert_attention_close

pytestmark = pytest.mark.gpu

DEV = "cuda"
PKV_ESCRATCH_TOO_SMALL = -7


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_52_gb300 import pagedkv
    pagedkv.get_device_error(clear=True)
    return pagedkv


def _noalloc_call(pk, w, kc, vc, out, max_len, pb):
    """The new entry point, called directly through the C ABI."""
    return pk.lib.pkv_paged_decode_attention_noalloc(
        ctypes.c_void_p(w.q.data_ptr()), w.num_seqs, w.q_heads, ctypes.c_void_p(kc.data_ptr()),
        ctypes.c_void_p(vc.data_ptr()), pk.cache_desc(kc),
        ctypes.c_void_p(w.block_tables.data_ptr()), w.block_tables.shape[1],
        ctypes.c_void_p(w.context_lens.data_ptr()), max_len, ctypes.c_float(w.scale),
        ctypes.c_void_p(out.data_ptr()), pb,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _workload(spec, lens):
    w = wl.make_decode_workload(spec, lens_override=lens)
    for n in ("q", "k_cache", "v_cache", "k_new", "v_new", "slot_mapping", "block_tables",
              "context_lens"):
        setattr(w, n, getattr(w, n).to(DEV))
    return w


@pytest.mark.parametrize("spec,lens,pb", [
    (wl.TINY, [17, 64, 100, 250], 2),                       # forced split, small scratch
    (wl.GQA_70B, [20000, 3000, 131, 9000], 0),               # automatic split plan
    (wl.MHA_7B, [4096, 600, 2222], 0),
])
def test_noalloc_matches_regular_entry_point_twice(pk, spec, lens, pb):
    w = _workload(spec, lens)
    kc, vc = w.k_cache, w.v_cache
    pk.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    max_len = max(lens)
    _, parts, need = pk.decode_plan(w.num_seqs, w.q_heads, w.kv_heads, w.d_head, max_len, pb)
    assert parts > 1 and 0 < need <= pk.lib.pkv_noalloc_scratch_bytes()
    ref = pk.paged_decode_attention(w.q, kc, vc, w.block_tables, w.context_lens, w.scale,
                                    max_context_len=max_len, partition_blocks=pb)
    outs = [torch.full_like(ref, float("nan")) for _ in range(4)]
    assert _noalloc_call(pk, w, kc, vc, outs[0], max_len, pb) == 0
    torch.cuda.synchronize()
    # after the first call (which loads the kernels and looks up the scratch
    # address), further calls take no device memory at all
    free_before, _ = torch.cuda.mem_get_info()
    for out in outs[1:]:                                      # more calls in a row
        assert _noalloc_call(pk, w, kc, vc, out, max_len, pb) == 0
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before
    for out in outs:
        assert_attention_close(out.cpu().numpy(), ref.cpu().numpy(), "no-alloc vs regular")
    assert pk.get_device_error() == 0


def test_noalloc_rejects_plans_beyond_the_scratch(pk):
    w = _workload(wl.TINY, [17, 64, 100, 250])
    out = torch.empty(w.num_seqs, w.q_heads, w.d_head, dtype=torch.float32, device=DEV)
    # 4 sequences claiming 8M-token contexts with 16-block partitions need far
    # more than the fixed scratch: rejected on the host, nothing launched
    big = 1 << 23
    _, _, need = pk.decode_plan(w.num_seqs, w.q_heads, w.kv_heads, w.d_head, big, 16)
    assert need > pk.lib.pkv_noalloc_scratch_bytes()
    assert _noalloc_call(pk, w, w.k_cache, w.v_cache, out, big, 16) == PKV_ESCRATCH_TOO_SMALL
    assert "scratch" in pk.status_string(PKV_ESCRATCH_TOO_SMALL)
