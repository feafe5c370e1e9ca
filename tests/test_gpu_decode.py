"""Paged decode attention on the GPU against the CPU oracle.

Small cases compare every output element; the full-size 7B-MHA, 70B-GQA and
128K long-context workloads run in the launch configuration the benchmark
times (automatic split plan) and compare every sequence of the batch.
"""

import numpy as np
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


def run_step(pk, w, partition_blocks=0, max_context_len=None):
    """One decode step on the GPU: append the new token of every sequence, then attend."""
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    pk.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    mcl = max(w.meta["lens"]) if max_context_len is None else max_context_len
    out = pk.paged_decode_attention(w.q, kc, vc, w.block_tables, w.context_lens, w.scale,
                                    max_context_len=mcl, partition_blocks=partition_blocks)
    torch.cuda.synchronize()
    return out


def _to_dev(w):
    for name in ("q", "k_cache", "v_cache", "k_new", "v_new", "slot_mapping", "block_tables",
                 "context_lens"):
        setattr(w, name, getattr(w, name).to(DEV))
    return w


@pytest.mark.parametrize("pb", [0, 1, 2, 3, 5, 16])
def test_tiny_config_all_partitions(pk, pb):
    w = wl.make_decode_workload(wl.TINY)
    ref = DecodeStepOracle(w, range(w.num_seqs)).output()
    out = run_step(pk, _to_dev(w), partition_blocks=pb)
    assert_attention_close(out.cpu().numpy(), ref, f"tiny pb={pb}")
    assert pk.get_device_error() == 0


SHAPES = [(8, 8, 128), (8, 4, 64), (16, 4, 128), (64, 8, 128), (32, 2, 64), (16, 16, 64)]
EDGE_LENS = [1, 15, 16, 17, 33, 200, 0, 161]


@pytest.mark.parametrize("hq,hkv,d", SHAPES + [(128, 8, 128)])
@pytest.mark.parametrize("pb", [0, 2])
def test_groups_heads_and_ragged_lengths(pk, hq, hkv, d, pb):
    spec = wl.DecodeSpec("edge", 11, len(EDGE_LENS), hq, hkv, d, lens=tuple(EDGE_LENS))
    w = wl.make_decode_workload(spec, lens_override=EDGE_LENS)
    # the empty sequence appends nothing
    w.slot_mapping[EDGE_LENS.index(0)] = -1
    ref = DecodeStepOracle(w, range(w.num_seqs)).output()
    out = run_step(pk, _to_dev(w), partition_blocks=pb)
    assert_attention_close(out.cpu().numpy(), ref, f"{hq}/{hkv} d{d} pb={pb}")
    assert np.all(out[EDGE_LENS.index(0)].cpu().numpy() == 0.0)
    assert pk.get_device_error() == 0


def test_massive_activation_outliers_small(pk):
    # the 70B-GQA recipe (0.1% K rows x100), shrunk to lengths the oracle does whole
    w = wl.make_decode_workload(wl.GQA_70B, lens_override=[1024, 3000, 777, 4096, 2049, 1500])
    ref = DecodeStepOracle(w, range(w.num_seqs)).output()
    for pb in (0, 7):
        out = run_step(pk, _to_dev(w) if not w.q.is_cuda else w, partition_blocks=pb)
        assert_attention_close(out.cpu().numpy(), ref, f"outliers pb={pb}")


def test_repeatable_bitwise(pk):
    w = _to_dev(wl.make_decode_workload(wl.GQA_70B, lens_override=[900, 2500, 64]))
    a = run_step(pk, w)
    b = run_step(pk, w)
    assert torch.equal(a, b)


def test_bad_block_id_and_context_are_flagged(pk):
    w = _to_dev(wl.make_decode_workload(wl.TINY))
    pk.get_device_error(clear=True)
    bt = w.block_tables.clone()
    bt[1, 0] = 10_000                      # outside the 64-block pool
    pk.paged_decode_attention(w.q, w.k_cache, w.v_cache, bt, w.context_lens, w.scale,
                              max_context_len=250)
    assert pk.get_device_error(clear=True) & 0x2
    lens = w.context_lens.clone()
    lens[0] = 16 * bt.shape[1] + 5         # longer than the block table
    out = pk.paged_decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables, lens, w.scale,
                                    max_context_len=int(lens.max()))
    assert pk.get_device_error(clear=True) & 0x4
    assert torch.isfinite(out).all()
    # a max_context_len below the real lengths: flagged, never out of bounds
    pk.paged_decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                              w.scale, max_context_len=40, partition_blocks=1)
    assert pk.get_device_error(clear=True) & 0x4


@pytest.mark.parametrize("name", ["mha7b", "gqa70b", "long128k"])
def test_full_size_configs_whole_batch(pk, name):
    # the benchmark's launch configuration (automatic split plan), every
    # sequence of the batch compared with the oracle
    spec = wl.DECODE_SPECS[name]
    w = wl.make_decode_workload(spec, device=DEV, gen_device=DEV)
    seqs = list(range(w.num_seqs))
    ref = DecodeStepOracle(w, seqs).output()
    out = run_step(pk, w)
    assert_attention_close(out.cpu().numpy(), ref, name)
    assert torch.isfinite(out).all()
    assert pk.get_device_error() == 0
    del w
    torch.cuda.empty_cache()


def test_merge_output_alignment_forms_agree(pk):
    # the split-K merge writes float4 rows when out is 16-byte aligned and
    # one float per thread otherwise (the ABI asks only for 4-byte alignment);
    # both forms compute the same sums and divisions, so the same bits
    w = _to_dev(wl.make_decode_workload(wl.GQA_70B, lens_override=[1024, 3000, 777, 64]))
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    pk.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    S, hq, d = w.q.shape
    kw = dict(max_context_len=3000, partition_blocks=16)   # several partitions per sequence
    aligned = pk.paged_decode_attention(w.q, kc, vc, w.block_tables, w.context_lens, w.scale, **kw)
    buf = torch.full((S * hq * d + 1,), float("nan"), dtype=torch.float32, device=DEV)
    shifted = buf[1:].view(S, hq, d)                        # 4 bytes past a 16-byte boundary
    assert shifted.data_ptr() % 16 == 4
    pk.paged_decode_attention(w.q, kc, vc, w.block_tables, w.context_lens, w.scale, out=shifted,
                              **kw)
    torch.cuda.synchronize()
    assert torch.equal(aligned, shifted)
    ref = DecodeStepOracle(w, range(S)).output()
    assert_attention_close(shifted.cpu().numpy(), ref, "merge, 4-byte aligned out")
    assert pk.get_device_error(clear=True) == 0


# ---- the length-balanced work list (partition_blocks = SPLIT_BALANCED, and
# the library's choice for batches with at most 2 x SMs (sequence, KV head)
# pairs): runs of near-equal size cut from the actual lengths on the device
LIST_LENS = [0, 1, 15, 16, 17, 16 * 1000 + 1, 4096, 33, 200, 16 * 64 + 1]


@pytest.mark.parametrize("hq,hkv,d", SHAPES)
def test_balanced_list_ragged_lengths(pk, hq, hkv, d):
    spec = wl.DecodeSpec("list", 13, len(LIST_LENS), hq, hkv, d, lens=tuple(LIST_LENS))
    w = wl.make_decode_workload(spec, lens_override=LIST_LENS)
    w.slot_mapping[LIST_LENS.index(0)] = -1          # the empty sequence appends nothing
    ref = DecodeStepOracle(w, range(w.num_seqs)).output()
    w = _to_dev(w)
    assert pk.decode_plan_uses_list(w.num_seqs, hq, hkv, d, max(LIST_LENS), pk.SPLIT_BALANCED)
    out = run_step(pk, w, partition_blocks=pk.SPLIT_BALANCED)
    assert_attention_close(out.cpu().numpy(), ref, f"list {hq}/{hkv} d{d}")
    assert np.all(out[LIST_LENS.index(0)].cpu().numpy() == 0.0)
    uni = run_step(pk, w, partition_blocks=pk.SPLIT_UNIFORM)
    assert_attention_close(uni.cpu().numpy(), ref, f"uniform {hq}/{hkv} d{d}")
    assert pk.get_device_error() == 0


@pytest.mark.parametrize("num_seqs", [1, 8, 16, 32])
def test_balanced_list_small_batches(pk, num_seqs):
    # 70B-GQA recipe at small batch sizes (outlier rows included), the list
    # compared whole with the oracle; the library's own choice is uniform
    w = wl.make_decode_workload(wl.GQA_70B, device=DEV, gen_device=DEV,
                                num_seqs_override=num_seqs)
    max_len = max(w.meta["lens"])
    assert pk.decode_plan_uses_list(num_seqs, 64, 8, 128, max_len, pk.SPLIT_BALANCED)
    assert not pk.decode_plan_uses_list(num_seqs, 64, 8, 128, max_len, 0)
    ref = DecodeStepOracle(w, range(num_seqs)).output()
    out = run_step(pk, w, partition_blocks=pk.SPLIT_BALANCED)
    assert_attention_close(out.cpu().numpy(), ref, f"list, {num_seqs} sequences")
    assert pk.get_device_error() == 0


def test_balanced_list_bad_context_and_workspace_fallback(pk):
    w = _to_dev(wl.make_decode_workload(wl.TINY))
    pk.get_device_error(clear=True)
    lens = w.context_lens.clone()
    lens[0] = 16 * w.block_tables.shape[1] + 5           # longer than the block table
    out = pk.paged_decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables, lens, w.scale,
                                    max_context_len=int(lens.max()),
                                    partition_blocks=pk.SPLIT_BALANCED)
    assert pk.get_device_error(clear=True) & 0x4
    assert torch.isfinite(out).all()
    # the library's choice (uniform) without a workspace: none needed here
    S, hq, d = w.q.shape
    ref = pk.paged_decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                    w.scale, max_context_len=250,
                                    partition_blocks=pk.SPLIT_UNIFORM)
    out2 = torch.empty_like(ref)
    st = pk.lib.pkv_paged_decode_attention_ex(
        pk._ptr(w.q), S, hq, pk._ptr(w.k_cache), pk._ptr(w.v_cache), pk.cache_desc(w.k_cache),
        pk._ptr(w.block_tables), w.block_tables.shape[1], pk._ptr(w.context_lens), 250,
        w.scale, pk._ptr(out2), pk._ptr(None), 0, 0, pk._stream(w.q))
    assert st == 0
    torch.cuda.synchronize()
    assert torch.equal(out2, ref)
    assert pk.get_device_error(clear=True) == 0


@pytest.mark.parametrize("max_ctas", [1, 7, 64, 300])
def test_limited_decode_matches_oracle(pk, max_ctas):
    # the balanced list on at most max_ctas CTAs, each looping over its runs
    lens = [5000, 17, 0, 1, 2600, 16 * 300 + 1, 900, 4096]
    w = wl.make_decode_workload(wl.GQA_70B, lens_override=lens)
    w.slot_mapping[lens.index(0)] = -1
    ref = DecodeStepOracle(w, range(len(lens))).output()
    w = _to_dev(w)
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    pk.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    out = pk.paged_decode_attention_limited(w.q, kc, vc, w.block_tables, w.context_lens,
                                            w.scale, max_ctas, max_context_len=max(lens))
    torch.cuda.synchronize()
    assert_attention_close(out.cpu().numpy(), ref, f"limited decode, {max_ctas} CTAs")
    assert np.all(out[lens.index(0)].cpu().numpy() == 0.0)
    assert pk.get_device_error() == 0


# ---- the decode step (pkv_paged_decode_step): append and attend, the append
# hidden under the attention; the same cache rows and outputs bit for bit


@pytest.mark.parametrize("name,lens", [("tiny", None), ("gqa70b", [1024, 3000, 777, 17, 16, 2049])])
def test_decode_step_equals_append_then_decode(pk, name, lens):
    spec = wl.DECODE_SPECS[name]
    w = _to_dev(wl.make_decode_workload(spec, lens_override=lens))
    mcl = max(w.meta["lens"])
    kc1, vc1 = w.k_cache.clone(), w.v_cache.clone()
    pk.kv_append(w.k_new, w.v_new, w.slot_mapping, kc1, vc1)
    sep = pk.paged_decode_attention(w.q, kc1, vc1, w.block_tables, w.context_lens, w.scale,
                                    max_context_len=mcl)
    kc2, vc2 = w.k_cache.clone(), w.v_cache.clone()
    fused = pk.paged_decode_step(w.q, w.k_new, w.v_new, w.slot_mapping, kc2, vc2,
                                 w.block_tables, w.context_lens, w.scale, max_context_len=mcl)
    torch.cuda.synchronize()
    assert torch.equal(kc1, kc2) and torch.equal(vc1, vc2)
    assert torch.equal(sep, fused)
    ref = DecodeStepOracle(_to_dev(wl.make_decode_workload(spec, lens_override=lens)),
                           range(w.num_seqs)).output()
    assert_attention_close(fused.cpu().numpy(), ref, f"decode step {name}")
    assert pk.get_device_error(clear=True) == 0


def test_decode_step_full_size_70b_gqa(pk):
    w = wl.make_decode_workload(wl.GQA_70B, device=DEV, gen_device=DEV)
    mcl = max(w.meta["lens"])
    sep = run_step(pk, w)
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    fused = pk.paged_decode_step(w.q, w.k_new, w.v_new, w.slot_mapping, kc, vc, w.block_tables,
                                 w.context_lens, w.scale, max_context_len=mcl)
    torch.cuda.synchronize()
    assert torch.equal(sep, fused)
    assert pk.get_device_error(clear=True) == 0


def test_decode_step_slot_elsewhere_is_flagged(pk):
    w = _to_dev(wl.make_decode_workload(wl.TINY))
    slots = w.slot_mapping.clone()
    slots[1] = -1                                  # no token appended: attends the cache as is
    slots[2] = int(w.block_tables[2, 0]) * 16 + 3  # an earlier position of sequence 2
    pk.get_device_error(clear=True)
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    pk.paged_decode_step(w.q, w.k_new, w.v_new, slots, kc, vc, w.block_tables, w.context_lens,
                         w.scale, max_context_len=250)
    torch.cuda.synchronize()
    assert pk.get_device_error(clear=True) == 0x1
