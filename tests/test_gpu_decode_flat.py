"""The flat split of the bf16 decode (partition_blocks = SPLIT_FLAT) against
the CPU oracle: the blocks of all sequences laid end to end are cut into
equal ranges, one per group of Hkv warps of a one-CTA-per-SM grid (warp h
of a group takes KV head h), so sequences are cut at arbitrary blocks, a
range crosses sequences, and a pair held by one group is written without
the merge.  Small cases compare every element; the 70B-GQA recipe at 1 to
64 sequences and at full size, 7B-MHA and the 128K contexts compare whole
batches."""

import numpy as np
import pytest
import torch

from paged_kv_cache_52_gb300 import workloads as wl
from parity import DecodeStepOracle, assert_attention_close
from test_gpu_decode import SHAPES, run_step, _to_dev

pytestmark = pytest.mark.gpu

DEV = "cuda"
FLAT_LENS = [0, 1, 15, 16, 17, 16 * 1000 + 1, 4096, 33, 200, 16 * 64 + 1, 0, 2]


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_52_gb300 import pagedkv
    pagedkv.get_device_error(clear=True)
    return pagedkv


@pytest.mark.parametrize("hq,hkv,d", SHAPES + [(128, 8, 128)])
def test_flat_ragged_lengths(pk, hq, hkv, d):
    spec = wl.DecodeSpec("flat", 17, len(FLAT_LENS), hq, hkv, d, lens=tuple(FLAT_LENS))
    w = wl.make_decode_workload(spec, lens_override=FLAT_LENS)
    for i, L in enumerate(FLAT_LENS):
        if L == 0:
            w.slot_mapping[i] = -1                     # an empty sequence appends nothing
    ref = DecodeStepOracle(w, range(w.num_seqs)).output()
    w = _to_dev(w)
    assert pk.decode_plan_uses_flat(w.num_seqs, hq, hkv, d, max(FLAT_LENS), pk.SPLIT_FLAT)
    out = run_step(pk, w, partition_blocks=pk.SPLIT_FLAT)
    assert_attention_close(out.cpu().numpy(), ref, f"flat {hq}/{hkv} d{d}")
    for i, L in enumerate(FLAT_LENS):
        if L == 0:
            assert np.all(out[i].cpu().numpy() == 0.0)
    assert pk.get_device_error() == 0


@pytest.mark.parametrize("d", [128, 64])
def test_flat_many_short_sequences(pk, d):
    # 700 sequences of 1..80 tokens: most ranges cross several sequences,
    # most pairs lie inside one group's range (written without the merge)
    lens = [1 + (i * 37) % 80 for i in range(700)]
    spec = wl.DecodeSpec("flat short", 18, len(lens), 16, 4, d, lens=tuple(lens))
    w = wl.make_decode_workload(spec, lens_override=lens)
    ref = DecodeStepOracle(w, range(w.num_seqs)).output()
    out = run_step(pk, _to_dev(w), partition_blocks=pk.SPLIT_FLAT)
    assert_attention_close(out.cpu().numpy(), ref, f"flat, 700 short sequences, d{d}")
    assert pk.get_device_error() == 0


@pytest.mark.parametrize("num_seqs", [1, 8, 16, 32, 64])
def test_flat_small_batches_70b_gqa(pk, num_seqs):
    w = wl.make_decode_workload(wl.GQA_70B, device=DEV, gen_device=DEV,
                                num_seqs_override=num_seqs)
    max_len = max(w.meta["lens"])
    assert pk.decode_plan_uses_flat(num_seqs, 64, 8, 128, max_len, pk.SPLIT_FLAT)
    ref = DecodeStepOracle(w, range(num_seqs)).output()
    out = run_step(pk, w, partition_blocks=pk.SPLIT_FLAT)
    assert_attention_close(out.cpu().numpy(), ref, f"flat, {num_seqs} sequences")
    assert pk.get_device_error() == 0


@pytest.mark.parametrize("name", ["gqa70b", "mha7b", "long128k"])
def test_flat_full_size_whole_batch(pk, name):
    spec = wl.DECODE_SPECS[name]
    w = wl.make_decode_workload(spec, device=DEV, gen_device=DEV)
    ref = DecodeStepOracle(w, range(w.num_seqs)).output()
    out = run_step(pk, w, partition_blocks=pk.SPLIT_FLAT)
    assert_attention_close(out.cpu().numpy(), ref, f"flat {name}")
    assert torch.isfinite(out).all()
    assert pk.get_device_error() == 0
    del w
    torch.cuda.empty_cache()


def test_flat_repeatable_and_bf16_out(pk):
    w = _to_dev(wl.make_decode_workload(wl.GQA_70B, lens_override=[900, 2500, 64, 1, 4097]))
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    pk.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    kw = dict(max_context_len=4097, partition_blocks=pk.SPLIT_FLAT)
    a = pk.paged_decode_attention(w.q, kc, vc, w.block_tables, w.context_lens, w.scale, **kw)
    b = pk.paged_decode_attention(w.q, kc, vc, w.block_tables, w.context_lens, w.scale, **kw)
    h = pk.paged_decode_attention(w.q, kc, vc, w.block_tables, w.context_lens, w.scale,
                                  out_dtype=torch.bfloat16, **kw)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert torch.equal(h, a.to(torch.bfloat16))          # the same result, rounded in the store
    assert pk.get_device_error(clear=True) == 0


def test_flat_bad_block_id_and_context_are_flagged(pk):
    w = _to_dev(wl.make_decode_workload(wl.TINY))
    pk.get_device_error(clear=True)
    bt = w.block_tables.clone()
    bt[1, 0] = 10_000                                    # outside the 64-block pool
    pk.paged_decode_attention(w.q, w.k_cache, w.v_cache, bt, w.context_lens, w.scale,
                              max_context_len=250, partition_blocks=pk.SPLIT_FLAT)
    assert pk.get_device_error(clear=True) & 0x2
    lens = w.context_lens.clone()
    lens[0] = 16 * bt.shape[1] + 5                       # longer than the block table
    out = pk.paged_decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables, lens, w.scale,
                                    max_context_len=int(lens.max()),
                                    partition_blocks=pk.SPLIT_FLAT)
    assert pk.get_device_error(clear=True) & 0x4
    assert torch.isfinite(out).all()
    lens[0] = -3                                         # negative: attended as empty
    out = pk.paged_decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables, lens, w.scale,
                                    max_context_len=250, partition_blocks=pk.SPLIT_FLAT)
    assert pk.get_device_error(clear=True) & 0x4
    assert torch.all(out[0] == 0)
    # a max_context_len below the real lengths: flagged, never out of bounds
    pk.paged_decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                              w.scale, max_context_len=40, partition_blocks=pk.SPLIT_FLAT)
    assert pk.get_device_error(clear=True) & 0x4


def test_flat_workspace_is_required_and_sized(pk):
    w = _to_dev(wl.make_decode_workload(wl.TINY))
    S, hq, d = w.q.shape
    _, _, ws = pk.decode_plan(S, hq, w.k_cache.shape[2], d, 250, pk.SPLIT_FLAT)
    assert ws > 0
    out = torch.empty(S, hq, d, dtype=torch.float32, device=DEV)
    small = torch.empty(ws - 1, dtype=torch.uint8, device=DEV)
    st = pk.lib.pkv_paged_decode_attention_ex(
        pk._ptr(w.q), S, hq, pk._ptr(w.k_cache), pk._ptr(w.v_cache), pk.cache_desc(w.k_cache),
        pk._ptr(w.block_tables), w.block_tables.shape[1], pk._ptr(w.context_lens), 250,
        w.scale, pk._ptr(out), pk._ptr(small), ws - 1, pk.SPLIT_FLAT, pk._stream(w.q))
    assert st == -4  # PKV_ENOMEM
    # more sequences than the flat split takes: refused when forced
    assert pk.lib.pkv_decode_plan_uses_flat(1025, 8, 8, 128, 256, pk.SPLIT_FLAT) < 0


def test_library_choice_takes_flat_for_mid_size_batches(pk):
    # 193 to 1024 (sequence, KV head) pairs at d_head 128 over bf16 pages
    for S, flat in ((8, False), (16, False), (24, False), (25, True), (64, True), (128, True),
                    (129, False), (256, False)):
        assert pk.decode_plan_uses_flat(S, 64, 8, 128, 8192, 0) == flat, S
    # the library's workspace at 16 sequences still covers the flat split,
    # which the FP8 decode takes there
    auto = pk.decode_plan(16, 64, 8, 128, 8192)[2]
    assert auto >= pk.decode_plan(16, 64, 8, 128, 8192, pk.SPLIT_FLAT)[2]
    assert not pk.decode_plan_uses_flat(32, 64, 8, 64, 8192, 0)      # measured at d 128 only


@pytest.mark.parametrize("num_seqs", [32, 48])
def test_decode_step_on_the_flat_split(pk, num_seqs):
    # the decode step with the library's choice (flat here): the append runs
    # beside the flat kernel, whose warps wait for it only before a
    # sequence's last page; cache rows and outputs equal append-then-decode
    w = wl.make_decode_workload(wl.GQA_70B, device=DEV, gen_device=DEV,
                                num_seqs_override=num_seqs)
    mcl = max(w.meta["lens"])
    assert pk.decode_plan_uses_flat(num_seqs, 64, 8, 128, mcl, 0)
    ref = DecodeStepOracle(w, range(num_seqs)).output()
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
    assert_attention_close(fused.cpu().numpy(), ref, f"decode step on the flat split, {num_seqs}")
    assert pk.get_device_error(clear=True) == 0

def test_decode_step_on_the_flat_split_skips_and_flags(pk):
    # 30 sequences on the flat split: one appends nothing (slot -1: it
    # attends the cache as is), one of length 1 (its last page is its first),
    # one whose slot lies in a block no sequence reads (flagged; the decode
    # attends the cache as is there too) -- equal to append-then-decode
    lens = [1200, 3000, 1, 700, 4096] + [500 + 97 * i for i in range(25)]
    w = _to_dev(wl.make_decode_workload(wl.GQA_70B, lens_override=lens))
    S = len(lens)
    assert pk.decode_plan_uses_flat(S, 64, 8, 128, max(lens), 0)
    slots = w.slot_mapping.clone()
    slots[1] = -1
    used = set(w.block_tables.flatten().tolist())
    spare = next(b for b in range(w.k_cache.shape[0]) if b not in used)
    slots[3] = spare * 16 + 5
    kc1, vc1 = w.k_cache.clone(), w.v_cache.clone()
    pk.kv_append(w.k_new, w.v_new, slots, kc1, vc1)
    sep = pk.paged_decode_attention(w.q, kc1, vc1, w.block_tables, w.context_lens, w.scale,
                                    max_context_len=max(lens))
    torch.cuda.synchronize()
    pk.get_device_error(clear=True)
    kc2, vc2 = w.k_cache.clone(), w.v_cache.clone()
    fused = pk.paged_decode_step(w.q, w.k_new, w.v_new, slots, kc2, vc2, w.block_tables,
                                 w.context_lens, w.scale, max_context_len=max(lens))
    torch.cuda.synchronize()
    assert pk.get_device_error(clear=True) == 0x1          # sequence 3's slot is elsewhere
    assert torch.equal(kc1, kc2) and torch.equal(vc1, vc2)
    assert torch.equal(sep, fused)
