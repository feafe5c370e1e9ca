"""The checked append on the GPU against the oracle's checked append: a slot
mapping without repeats is appended exactly as the plain append does; one
that names a slot twice leaves both caches bit for bit as they were and sets
the duplicate-slot bit of the device error word."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_52_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"
DUP_BIT = 0x80


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_52_gb300 import pagedkv
    pagedkv.get_device_error(clear=True)
    return pagedkv


def _run(pk, w, slots):
    kc, vc = w.k_cache.to(DEV), w.v_cache.to(DEV)
    ws = pk.kv_append_checked_workspace(kc)
    ws.fill_(0xAB)                                   # the call must clear what it uses
    pk.kv_append(w.k_new.to(DEV), w.v_new.to(DEV), torch.from_numpy(slots).to(DEV), kc, vc,
                 checked_workspace=ws)
    torch.cuda.synchronize()
    return wl.bf16_bits(kc), wl.bf16_bits(vc), pk.get_device_error(clear=True)


def _oracle(w, slots):
    return oracle.kv_append_checked(wl.bf16_bits(w.k_new), wl.bf16_bits(w.v_new), slots,
                                    wl.bf16_bits(w.k_cache), wl.bf16_bits(w.v_cache))


@pytest.mark.parametrize("case", ["unique", "skips", "repeat", "repeat_far"])
def test_checked_append_matches_oracle(pk, case):
    lens = [int(x) for x in np.random.default_rng(21).integers(1, 300, 24)]
    spec = wl.DecodeSpec("append", 17, 24, 8, 2, 64, lens=tuple(lens))
    w = wl.make_decode_workload(spec, lens_override=lens)
    slots = w.slot_mapping.numpy().copy()
    if case == "skips":
        slots[[2, 5, 9]] = -1                        # -1 repeats; not a duplicate
    elif case == "repeat":
        slots[7] = slots[6]
    elif case == "repeat_far":
        slots[23] = slots[0]                         # first and last token
    k_ref, v_ref, rejected = _oracle(w, slots)
    k_got, v_got, err = _run(pk, w, slots)
    assert np.array_equal(k_got, k_ref) and np.array_equal(v_got, v_ref)
    assert bool(err & DUP_BIT) == rejected
    assert rejected == case.startswith("repeat")
    assert err & ~DUP_BIT == 0


def test_checked_append_many_tokens_and_out_of_pool_slot(pk):
    # a mixed-step sized append (thousands of tokens across many blocks); a
    # slot outside the pool is skipped and flagged as by the plain append,
    # and does not count as a repeat
    w = wl.make_mixed_workload(device=DEV, gen_device=DEV, num_decode=32, num_prefill=2)
    slots = w.slot_mapping.cpu().numpy().copy()
    nb = w.k_cache.shape[0]
    bad = slots.copy()
    bad[10] = nb * 16 + 5
    kc, vc = w.k_cache.to(DEV), w.v_cache.to(DEV)
    ws = pk.kv_append_checked_workspace(kc)
    pk.kv_append(w.k_new.to(DEV), w.v_new.to(DEV), torch.from_numpy(bad).to(DEV), kc, vc,
                 checked_workspace=ws)
    torch.cuda.synchronize()
    err = pk.get_device_error(clear=True)
    assert err & 0x1 and not err & DUP_BIT
    keep = bad != nb * 16 + 5
    k_ref, v_ref = oracle.kv_append(wl.bf16_bits(w.k_new)[keep], wl.bf16_bits(w.v_new)[keep],
                                    bad[keep], wl.bf16_bits(w.k_cache), wl.bf16_bits(w.v_cache))
    assert np.array_equal(wl.bf16_bits(kc), k_ref) and np.array_equal(wl.bf16_bits(vc), v_ref)
