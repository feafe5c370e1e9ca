"""KV append on the GPU is bit-exact against the oracle on the whole pools
(so rows the step does not own keep their previous contents)."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_52_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_52_gb300 import pagedkv
    pagedkv.get_device_error(clear=True)
    return pagedkv


def _oracle_append(k_new, v_new, slots, kc, vc):
    return oracle.kv_append(wl.bf16_bits(k_new), wl.bf16_bits(v_new), np.asarray(slots),
                            wl.bf16_bits(kc), wl.bf16_bits(vc))


def _check(pk, k_new, v_new, slots, kc0, vc0):
    k_ref, v_ref = _oracle_append(k_new, v_new, slots.cpu().numpy(), kc0, vc0)
    kc, vc = kc0.to(DEV), vc0.to(DEV)
    pk.kv_append(k_new.to(DEV) if not k_new.is_cuda else k_new,
                 v_new.to(DEV) if not v_new.is_cuda else v_new, slots.to(DEV), kc, vc)
    torch.cuda.synchronize()
    assert np.array_equal(wl.bf16_bits(kc), k_ref)
    assert np.array_equal(wl.bf16_bits(vc), v_ref)


def test_append_tiny_config(pk):
    w = wl.make_decode_workload(wl.TINY)
    _check(pk, w.k_new, w.v_new, w.slot_mapping, w.k_cache, w.v_cache)
    assert pk.get_device_error() == 0


def test_append_skip_slots_and_fused_qkv_views(pk):
    w = wl.make_mixed_workload(num_prefill=3, num_decode=5, chunk=37, prior_range=(0, 60),
                               shared_prefix=32, decode_cap=300)
    T, hkv, d = w.k_new.shape
    hq = 64
    # k, v as strided views of one fused [T, (Hq + 2 Hkv) * d] projection output
    g = torch.Generator().manual_seed(9)
    fused = torch.randn(T, (hq + 2 * hkv) * d, generator=g).to(torch.bfloat16)
    fused[:, hq * d:(hq + hkv) * d] = w.k_new.reshape(T, -1)
    fused[:, (hq + hkv) * d:] = w.v_new.reshape(T, -1)
    fused_dev = fused.to(DEV)
    k_view = fused_dev[:, hq * d:(hq + hkv) * d].view(T, hkv, d)
    v_view = fused_dev[:, (hq + hkv) * d:].view(T, hkv, d)
    assert k_view.stride(0) == (hq + 2 * hkv) * d
    slots = w.slot_mapping.clone()
    slots[::7] = -1
    _check(pk, k_view, v_view, slots, w.k_cache, w.v_cache)
    assert pk.get_device_error() == 0


def test_append_bulk_many_tokens(pk):
    # 4344 tokens of the mixed-step shape (8 x 512 prefill rows + 248 decode rows)
    w = wl.make_mixed_workload(num_prefill=8, num_decode=248, chunk=512, prior_range=(0, 64),
                               shared_prefix=16, decode_cap=200)
    assert w.slot_mapping.shape[0] == 8 * 512 + 248
    _check(pk, w.k_new, w.v_new, w.slot_mapping, w.k_cache, w.v_cache)


def test_append_out_of_range_slot_is_skipped_and_flagged(pk):
    w = wl.make_decode_workload(wl.TINY)
    nslots = w.k_cache.shape[0] * w.k_cache.shape[1]
    slots = w.slot_mapping.clone()
    slots[2] = nslots          # past the pool
    slots[3] = -5              # negative but not -1
    pk.get_device_error(clear=True)
    ref_slots = slots.clone()
    ref_slots[2] = -1
    ref_slots[3] = -1
    k_ref, v_ref = _oracle_append(w.k_new, w.v_new, ref_slots.numpy(), w.k_cache, w.v_cache)
    kc, vc = w.k_cache.to(DEV), w.v_cache.to(DEV)
    pk.kv_append(w.k_new.to(DEV), w.v_new.to(DEV), slots.to(DEV), kc, vc)
    assert pk.get_device_error() & 0x1
    assert np.array_equal(wl.bf16_bits(kc), k_ref)
    assert np.array_equal(wl.bf16_bits(vc), v_ref)


def test_append_zero_tokens_is_a_no_op(pk):
    w = wl.make_decode_workload(wl.TINY)
    kc = w.k_cache.to(DEV)
    vc = w.v_cache.to(DEV)
    empty = torch.empty(0, *w.k_new.shape[1:], dtype=torch.bfloat16, device=DEV)
    pk.kv_append(empty, empty, torch.empty(0, dtype=torch.int64, device=DEV), kc, vc)
    assert np.array_equal(wl.bf16_bits(kc), wl.bf16_bits(w.k_cache))
