"""Chunked-prefill attention (tcgen05 + TMEM kernel) against the CPU oracle,
and the continuous-batching mixed step (append, prefill chunks, decodes)."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_52_gb300 import workloads as wl
from parity import DecodeStepOracle, PrefillStepOracle, assert_attention_close

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_52_gb300 import pagedkv
    pagedkv.get_device_error(clear=True)
    return pagedkv


def _to_dev(w):
    for n in ("k_cache", "v_cache", "k_new", "v_new", "slot_mapping", "q_prefill", "q_start",
              "prefill_tables", "prefill_lens", "q_decode", "decode_tables", "decode_lens"):
        setattr(w, n, getattr(w, n).to(DEV))
    return w


def run_prefill(pk, w, causal=True, max_q_len=None):
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    pk.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    out = torch.full((w.q_prefill.shape[0], w.q_prefill.shape[1], w.q_prefill.shape[2]),
                     float("nan"), dtype=torch.float32, device=DEV)
    mql = max(w.meta.get("chunks", [w.meta.get("chunk", 0)])) if max_q_len is None else max_q_len
    pk.paged_prefill_attention(w.q_prefill, w.q_start, kc, vc, w.prefill_tables, w.prefill_lens,
                               causal, w.scale, out=out, max_q_len=mql)
    torch.cuda.synchronize()
    return out, kc, vc


PRIORS = [0, 40, 17, 300, 1000, 5]
CHUNKS = [5, 130, 1, 129, 64, 16]
SHAPES = [(8, 8, 128), (8, 4, 64), (16, 4, 128), (64, 8, 128), (32, 2, 64), (16, 16, 64)]


@pytest.mark.parametrize("hq,hkv,d", SHAPES)
@pytest.mark.parametrize("causal", [True, False])
def test_chunks_groups_and_ragged_lengths(pk, hq, hkv, d, causal):
    w = wl.make_chunked_workload(hq, hkv, d, PRIORS, CHUNKS)
    ref = PrefillStepOracle(w, range(len(CHUNKS)), causal=causal).output()
    out, _, _ = run_prefill(pk, _to_dev(w), causal=causal)
    assert_attention_close(out.cpu().numpy(), ref, f"{hq}/{hkv} d{d} causal={causal}")
    assert pk.get_device_error() == 0


def test_long_chunk_many_kv_tiles(pk):
    # 2 chunks spanning several query tiles and ~40 K/V tiles (rescaling path)
    w = wl.make_chunked_workload(64, 8, 128, [4000, 700], [300, 513], config_id=7)
    ref = PrefillStepOracle(w, [0, 1]).output()
    out, _, _ = run_prefill(pk, _to_dev(w))
    assert_attention_close(out.cpu().numpy(), ref, "long chunk")


def test_outlier_keys_in_prefill(pk):
    # massive-activation K rows (x100) force many lazy-rescale events
    w = wl.make_chunked_workload(64, 8, 128, [900, 64], [200, 77], config_id=8)
    g = torch.Generator().manual_seed(5)
    kc = w.k_cache.float()
    rows = torch.randperm(kc.shape[0] * 16, generator=g)[:40]
    kc.view(-1, 8, 128)[rows] *= 100.0
    w.k_cache = kc.to(torch.bfloat16)
    ref = PrefillStepOracle(w, [0, 1]).output()
    out, _, _ = run_prefill(pk, _to_dev(w))
    assert_attention_close(out.cpu().numpy(), ref, "outliers")


def test_shared_prefix_mixed_step_small(pk):
    w = _to_dev(wl.make_mixed_workload(num_prefill=3, num_decode=5, chunk=200,
                                       prior_range=(0, 300), shared_prefix=64, decode_cap=700))
    pre_ref = PrefillStepOracle(w, range(3)).output()
    # decode oracle: the decodes' appended rows are the last 5 of k_new
    out, kc, vc = run_prefill(pk, w, max_q_len=200)
    assert_attention_close(out.cpu().numpy(), pre_ref, "mixed prefill")
    dec = pk.paged_decode_attention(w.q_decode, kc, vc, w.decode_tables, w.decode_lens, w.scale,
                                    max_context_len=max(w.meta["decode_lens"]))
    torch.cuda.synchronize()
    P = 3 * 200
    dw = wl.DecodeWorkload("mixed decodes", w.q_decode, w.k_cache, w.v_cache, w.k_new[P:],
                           w.v_new[P:], w.slot_mapping[P:], w.decode_tables, w.decode_lens,
                           w.scale, {"lens": w.meta["decode_lens"]})
    # the prefill chunks' rows are appended too; the decodes never read them
    dref = DecodeStepOracle(dw, range(5)).output()
    assert_attention_close(dec.cpu().numpy(), dref, "mixed decode")


def test_repeatable_bitwise(pk):
    w = _to_dev(wl.make_chunked_workload(64, 8, 128, [500, 0], [300, 77], config_id=9))
    a, _, _ = run_prefill(pk, w)
    b, _, _ = run_prefill(pk, w)
    assert torch.equal(a, b)


def test_bad_query_range_is_flagged(pk):
    w = _to_dev(wl.make_chunked_workload(16, 4, 64, [10, 20], [8, 8], config_id=10))
    pk.get_device_error(clear=True)
    lens = w.prefill_lens.clone()
    lens[1] = 4                       # chunk of 8 longer than its context
    out = torch.zeros(w.q_prefill.shape, dtype=torch.float32, device=DEV)
    pk.paged_prefill_attention(w.q_prefill, w.q_start, w.k_cache, w.v_cache, w.prefill_tables,
                               lens, True, w.scale, out=out, max_q_len=8)
    assert pk.get_device_error(clear=True) & 0x10
    assert torch.all(out[8:] == 0)    # the bad sequence is skipped
    assert torch.any(out[:8] != 0)    # the good one is computed
    # chunks of 8 with max_q_len 4: both sequences are rejected whole (no row
    # is written), and the stream-ordered query reports a failed check
    out.zero_()
    pk.paged_prefill_attention(w.q_prefill, w.q_start, w.k_cache, w.v_cache, w.prefill_tables,
                               w.prefill_lens, True, w.scale, out=out, max_q_len=4)
    status, bits = pk.get_last_device_error()
    assert status == pk.PKV_EDEVICE_CHECK and bits & 0x10
    assert torch.all(out == 0)
    assert pk.get_last_device_error() == (0, 0)


# query-token ranges of the first, a middle and the last 128-row tile (16
# tokens x the 8 heads of the group) of a 512-token chunk
MIXED_TILES = [(0, 16), (240, 256), (496, 512)]


def mixed_prefill_tiles_close(out, w, what):
    """The first, a middle and the last query tile of every chunk of the
    mixed step against the oracle."""
    orc = PrefillStepOracle(w, range(len(w.meta["prefill_lens"])))
    qs = w.q_start.cpu().numpy()
    for si in range(len(orc.seqs)):
        for a, b in MIXED_TILES:
            ref = orc.token_range_output(si, a, b)
            got = out[int(qs[si]) + a:int(qs[si]) + b].cpu().numpy()
            assert_attention_close(got, ref, f"{what}: chunk {si} tokens [{a}, {b})")


def test_full_mixed_step(pk):
    """The 70B-GQA continuous-batching step at full size: append 8 x 512 + 248
    tokens, prefill the 8 chunks, decode the 248 sequences.  Every decode and
    three query tiles of every chunk are compared with the oracle."""
    w = wl.make_mixed_workload(device=DEV, gen_device=DEV)
    P = 8 * 512
    dw = wl.DecodeWorkload("mixed decodes", w.q_decode, w.k_cache, w.v_cache, w.k_new[P:],
                           w.v_new[P:], w.slot_mapping[P:], w.decode_tables, w.decode_lens,
                           w.scale, {"lens": w.meta["decode_lens"]})
    dor = DecodeStepOracle(dw, range(dw.q.shape[0]))
    out, kc, vc = run_prefill(pk, w, max_q_len=512)
    dec = pk.paged_decode_attention(w.q_decode, kc, vc, w.decode_tables, w.decode_lens, w.scale,
                                    max_context_len=max(w.meta["decode_lens"]))
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    mixed_prefill_tiles_close(out, w, "mixed prefill (bf16 hi + lo P)")  # w's pools are unchanged
    assert_attention_close(dec.cpu().numpy(), dor.output(), "mixed decodes")
    assert pk.get_device_error() == 0


def test_non_causal_chunk_longer_than_context(pk):
    # without the causal mask a chunk may hold more queries than the context has keys
    w = wl.make_chunked_workload(16, 4, 128, [0, 0], [40, 7], config_id=14)
    lens = torch.tensor([25, 3], dtype=torch.int32)          # fewer keys than queries
    w.prefill_lens = lens
    ref = oracle.paged_prefill_attention(
        wl.bf16_bits(w.q_prefill), w.q_start.numpy(), wl.bf16_bits(w.k_cache),
        wl.bf16_bits(w.v_cache), w.prefill_tables.numpy(), lens.numpy(), False, w.scale)
    w = _to_dev(w)
    out = torch.full(w.q_prefill.shape, float("nan"), dtype=torch.float32, device=DEV)
    pk.paged_prefill_attention(w.q_prefill, w.q_start, w.k_cache, w.v_cache, w.prefill_tables,
                               w.prefill_lens, False, w.scale, out=out, max_q_len=40)
    torch.cuda.synchronize()
    assert_attention_close(out.cpu().numpy(), ref, "non-causal n > context")
    assert pk.get_device_error() == 0


@pytest.mark.parametrize("key", [40, 100, 140, 197])
@pytest.mark.parametrize("workspace", [False, True])
def test_running_max_jump_inside_a_tile(pk, key, workspace):
    # The kernel takes the exponentials against the running max with no max
    # pass and checks the sums (each 64-key group's on the plain path, the
    # tile's rounded sum on the workspace path); a key whose score jumps far
    # above that max fails the check.  The first 128-key tile seeds the max
    # from its first 32 keys: keys 40 and 100 lie beyond them in that tile,
    # so its check fails and it takes the two-pass path.  Key 140 sits in the
    # first group of the second tile (recomputed with the max pass), key 197
    # in its second group, after the first group was stored (on the plain
    # path its P, O and the row sum are rescaled in place).  All must match
    # the oracle.
    w = wl.make_chunked_workload(64, 8, 128, [300], [64], config_id=21)
    rows = w.k_cache.view(-1, 8, 128)
    tables = w.prefill_tables.numpy()
    slot = int(tables[0, key // 16]) * 16 + key % 16
    rows[slot] = (rows[slot].float() * 100.0).to(torch.bfloat16)
    ref = PrefillStepOracle(w, [0]).output()
    wd = _to_dev(w)
    if workspace:
        kc, vc = wd.k_cache.clone(), wd.v_cache.clone()
        pk.kv_append(wd.k_new, wd.v_new, wd.slot_mapping, kc, vc)
        ws = pk.prefill_workspace(1, wd.prefill_tables.shape[1], 8, 128, DEV)
        out = pk.paged_prefill_attention(wd.q_prefill, wd.q_start, kc, vc, wd.prefill_tables,
                                         wd.prefill_lens, True, wd.scale, max_q_len=64,
                                         workspace=ws)
        torch.cuda.synchronize()
    else:
        out, _, _ = run_prefill(pk, wd, max_q_len=64)
    assert_attention_close(out.cpu().numpy(), ref, f"max jump at key {key}")
    assert pk.get_device_error(clear=True) == 0
