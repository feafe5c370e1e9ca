"""The continuous-batching step's attention in one persistent launch
(pkv_mixed_step_attention) against the CPU oracle: its prefill outputs equal
the workspace prefill's bit for bit (the same tile arithmetic), and both its
prefill and its decode outputs match the oracle."""

import dataclasses

import numpy as np
import pytest
import torch

from paged_kv_cache_52_gb300 import workloads as wl
from parity import DecodeStepOracle, PrefillStepOracle, assert_attention_close
from test_gpu_prefill import mixed_prefill_tiles_close

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_52_gb300 import pagedkv
    pagedkv.get_device_error(clear=True)
    return pagedkv


def _decode_view(w):
    """The decode half of a mixed workload as a decode step."""
    P = len(w.meta["prefill_lens"]) * w.meta["chunk"]
    return wl.DecodeWorkload("mixed decodes", w.q_decode, w.k_cache, w.v_cache, w.k_new[P:],
                             w.v_new[P:], w.slot_mapping[P:], w.decode_tables, w.decode_lens,
                             w.scale, {"lens": w.meta["decode_lens"]})


def _run(pk, w):
    """Append every new token, then the fused step; also the workspace
    prefill on the same pools for the bitwise comparison."""
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    pk.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    chunk = w.meta["chunk"]
    mdl = max(w.meta["decode_lens"])
    pout, dout = pk.mixed_step_attention(w.q_prefill, w.q_start, w.prefill_tables, w.prefill_lens,
                                         True, w.q_decode, w.decode_tables, w.decode_lens, kc, vc,
                                         w.scale, chunk, mdl)
    ws = pk.prefill_workspace(w.prefill_lens.shape[0], w.prefill_tables.shape[1], kc.shape[2],
                              kc.shape[3], kc.device)
    sep = pk.paged_prefill_attention(w.q_prefill, w.q_start, kc, vc, w.prefill_tables,
                                     w.prefill_lens, True, w.scale, max_q_len=chunk, workspace=ws)
    torch.cuda.synchronize()
    return pout, dout, sep


SMALL = dataclasses.replace(wl.MIXED, name="small mixed step", config_id=21, num_prefill=3,
                            chunk=96, prior_range=(0, 700), num_decode=37, decode_median=500.0,
                            max_len=6000, shared_prefix=64)


@pytest.mark.parametrize("hq,hkv,d", [(64, 8, 128), (16, 4, 64), (8, 8, 128), (32, 2, 64)])
def test_mixed_step_small_matches_oracle_and_separate_prefill(pk, hq, hkv, d):
    spec = dataclasses.replace(SMALL, q_heads=hq, kv_heads=hkv, d_head=d)
    w = wl.make_mixed_workload(spec)
    pre = PrefillStepOracle(w, range(spec.num_prefill)).output()
    dec = DecodeStepOracle(_decode_view(w), range(spec.num_decode)).output()
    for n in ("k_cache", "v_cache", "k_new", "v_new", "slot_mapping", "q_prefill", "q_start",
              "prefill_tables", "prefill_lens", "q_decode", "decode_tables", "decode_lens"):
        setattr(w, n, getattr(w, n).to(DEV))
    pout, dout, sep = _run(pk, w)
    assert torch.equal(pout, sep)
    assert_attention_close(pout.cpu().numpy(), pre, f"mixed prefill {hq}/{hkv} d{d}")
    assert_attention_close(dout.cpu().numpy(), dec, f"mixed decode {hq}/{hkv} d{d}")
    assert pk.get_device_error(clear=True) == 0


def test_mixed_step_full_size(pk):
    """The 70B-GQA mixed step (8 chunks of 512 + 248 decodes): every decode
    and three query tiles of every chunk against the oracle, the whole
    prefill output against the workspace prefill bit for bit."""
    w = wl.make_mixed_workload(device=DEV, gen_device=DEV)
    dor = DecodeStepOracle(_decode_view(w), range(w.q_decode.shape[0]))
    pout, dout, sep = _run(pk, w)
    assert torch.equal(pout, sep)
    mixed_prefill_tiles_close(pout, w, "fused mixed step, prefill")
    assert_attention_close(dout.cpu().numpy(), dor.output(), "fused mixed step, decodes")
    assert pk.get_device_error(clear=True) == 0


def test_mixed_step_repeatable(pk):
    w = wl.make_mixed_workload(SMALL, device=DEV, gen_device=DEV)
    a = _run(pk, w)
    b = _run(pk, w)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def _run_groups(pk, w, gs, gp, span=0):
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    pk.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    chunk = w.meta["chunk"]
    mdl = max(w.meta["decode_lens"])
    sizes = (gs[1:] - gs[:-1]).tolist()
    pout, dout = pk.mixed_step_attention(
        w.q_prefill, w.q_start, w.prefill_tables, w.prefill_lens, True, w.q_decode,
        w.decode_tables, w.decode_lens, kc, vc, w.scale, chunk, mdl, prefill_span_permille=span,
        decode_groups=(gs.to(DEV), gp.to(DEV), max(sizes), int(gp.max())))
    torch.cuda.synchronize()
    return pout, dout


@pytest.mark.parametrize("hq,hkv,d", [(64, 8, 128), (16, 4, 64)])
def test_mixed_step_prefix_groups_small(pk, hq, hkv, d):
    # four decode groups over the shared 4-block prefix (one of them claims
    # only its first 2 blocks), one decode outside every group, and one member
    # whose third prefix page is a private copy: flagged, decoded whole
    spec = dataclasses.replace(SMALL, q_heads=hq, kv_heads=hkv, d_head=d)
    w = wl.make_mixed_workload(spec)
    used = set(w.prefill_tables.flatten().tolist()) | set(w.decode_tables.flatten().tolist())
    spare = next(b for b in range(w.meta["num_blocks"]) if b not in used)
    w.decode_tables[12, 2] = spare                       # member of group 1
    gs = torch.tensor([0, 10, 25, 30, 36], dtype=torch.int32)   # decode 36 has no group
    gp = torch.tensor([4, 4, 2, 4], dtype=torch.int32)
    pre = PrefillStepOracle(w, range(spec.num_prefill)).output()
    dec = DecodeStepOracle(_decode_view(w), range(spec.num_decode)).output()
    for n in ("k_cache", "v_cache", "k_new", "v_new", "slot_mapping", "q_prefill", "q_start",
              "prefill_tables", "prefill_lens", "q_decode", "decode_tables", "decode_lens"):
        setattr(w, n, getattr(w, n).to(DEV))
    pk.get_device_error(clear=True)
    pout, dout = _run_groups(pk, w, gs, gp)
    assert pk.get_device_error(clear=True) == 0x100      # the mismatched member
    assert_attention_close(pout.cpu().numpy(), pre, f"grouped mixed prefill {hq}/{hkv} d{d}")
    assert_attention_close(dout.cpu().numpy(), dec, f"grouped mixed decode {hq}/{hkv} d{d}")


def test_mixed_step_prefix_group_full_size(pk):
    # the 70B-GQA mixed step with its 248 decodes as one group sharing the
    # 1024-token prefix: every decode against the oracle, the prefill bit for
    # bit against the workspace prefill
    w = wl.make_mixed_workload(device=DEV, gen_device=DEV)
    S = w.q_decode.shape[0]
    dor = DecodeStepOracle(_decode_view(w), range(S))
    gs = torch.tensor([0, S], dtype=torch.int32)
    gp = torch.tensor([w.meta["shared_prefix"] // 16], dtype=torch.int32)
    pout, dout = _run_groups(pk, w, gs, gp)
    _, _, sep = _run(pk, w)
    assert torch.equal(pout, sep)
    assert_attention_close(dout.cpu().numpy(), dor.output(), "fused mixed step with prefix group")
    assert pk.get_device_error(clear=True) == 0
