"""Pins of the CPU oracle to facts fixed by the pages and by mathematics.

None of these checks re-derives the oracle from itself: each compares it with
a worked value printed on the pages, a closed form, a library routine
(torch's scaled_dot_product_attention in float64), an invariance the pages
state (paging is pure address translation; pages may sit anywhere), or a
brute-force recomputation.  The mutation tests at the end plant plausible
mistakes into copies of the oracle's attention and check that the pins catch
them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import paged_attention as opa
from paged_kv_cache_52_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _f64(t):
    return oracle.bf16_bits_to_f64(wl.bf16_bits(t))


# ---------------------------------------------------------------------------
# bf16 handling against torch's own conversion (library routine)
# ---------------------------------------------------------------------------
def test_bf16_widen_and_round_match_torch():
    g = torch.Generator().manual_seed(3)
    x = torch.randn(100_000, generator=g, dtype=torch.float32) * torch.exp(
        torch.randn(100_000, generator=g) * 4)
    t_bf16 = x.to(torch.bfloat16)
    bits = wl.bf16_bits(t_bf16)
    assert np.array_equal(oracle.f64_to_bf16_bits(x.numpy().astype(np.float64)), bits)
    assert np.array_equal(oracle.bf16_bits_to_f64(bits), t_bf16.to(torch.float64).numpy())


# ---------------------------------------------------------------------------
# Byte formula: worked values on the pages (tests/golden/kv_bytes.json)
# ---------------------------------------------------------------------------
def test_kv_byte_formula_matches_worked_values():
    gold = _golden("kv_bytes.json")
    for case in gold["cases"]:
        per_tok = oracle.kv_bytes_per_token(case["num_layers"], case["kv_heads"],
                                            case["d_head"], case["dtype_size"])
        if "bytes_per_token" in case:
            assert per_tok == case["bytes_per_token"], case["cite"]
        if "total_gib" in case:
            assert per_tok * case["seq_len"] == case["total_gib"] * 2 ** 30, case["cite"]
    p3 = gold["p3_formula"]
    S, K, H, L = p3["S"], p3["K"], p3["H"], p3["L"]
    assert S * oracle.kv_bytes_per_token(L, K, H, 2) == 4 * S * K * H * L
    # one layer's pool tensor [2, NB, bs, Hkv, d] (nano-vLLM pool shape)
    nb, bs = 1000, 16
    assert oracle.kv_cache_bytes(nb, bs, 8, 128, 2) == \
        nb * bs * oracle.kv_bytes_per_token_per_layer(8, 128, 2)
    assert oracle.kv_cache_bytes(nb, bs, 8, 128, 2) == \
        torch.empty(2, nb, bs, 8, 128, dtype=torch.bfloat16).nbytes


# ---------------------------------------------------------------------------
# Append: brute force through the flat row view, bit-exact, canary rows kept
# ---------------------------------------------------------------------------
def test_append_matches_flat_row_brute_force():
    w = wl.make_decode_workload(wl.TINY)
    kc, vc = wl.bf16_bits(w.k_cache), wl.bf16_bits(w.v_cache)
    kn, vn = wl.bf16_bits(w.k_new), wl.bf16_bits(w.v_new)
    slots = w.slot_mapping.numpy().copy()
    slots[1] = -1                                     # one token skipped
    k_out, v_out = oracle.kv_append(kn, vn, slots, kc, vc)
    nb, bs, hkv, d = kc.shape
    exp_k = kc.reshape(nb * bs, hkv, d).copy()        # row-major: slot = flat row
    exp_v = vc.reshape(nb * bs, hkv, d).copy()
    for t, s in enumerate(slots):
        if s >= 0:
            exp_k[s] = kn[t]
            exp_v[s] = vn[t]
    assert np.array_equal(k_out.reshape(nb * bs, hkv, d), exp_k)
    assert np.array_equal(v_out.reshape(nb * bs, hkv, d), exp_v)
    changed = np.any(k_out.reshape(nb * bs, -1) != kc.reshape(nb * bs, -1), axis=1)
    assert set(np.nonzero(changed)[0].tolist()) <= {int(s) for s in slots if s >= 0}
    assert not changed[w.slot_mapping.numpy()[1]] or slots[1] != -1
    with pytest.raises(ValueError):
        oracle.kv_append(kn[:1], vn[:1], np.array([nb * bs]), kc, vc)


def test_checked_append_rejects_a_repeated_slot():
    # every token owns its row: a mapping that names one row twice is
    # rejected whole (caches unchanged); -1 may repeat freely
    w = wl.make_decode_workload(wl.TINY)
    kc, vc = wl.bf16_bits(w.k_cache), wl.bf16_bits(w.v_cache)
    kn, vn = wl.bf16_bits(w.k_new), wl.bf16_bits(w.v_new)
    slots = w.slot_mapping.numpy().copy()
    nb, bs, hkv, d = kc.shape
    k1, v1, rej = oracle.kv_append_checked(kn, vn, slots, kc, vc)
    assert not rej
    exp_k = kc.reshape(nb * bs, hkv, d).copy()
    exp_v = vc.reshape(nb * bs, hkv, d).copy()
    for t, s_ in enumerate(slots):
        exp_k[s_] = kn[t]
        exp_v[s_] = vn[t]
    assert np.array_equal(k1.reshape(nb * bs, hkv, d), exp_k)
    assert np.array_equal(v1.reshape(nb * bs, hkv, d), exp_v)
    dup = slots.copy()
    dup[3] = dup[0]                                   # two tokens, one row
    k2, v2, rej = oracle.kv_append_checked(kn, vn, dup, kc, vc)
    assert rej and np.array_equal(k2, kc) and np.array_equal(v2, vc)
    skips = slots.copy()
    skips[1] = skips[2] = -1                          # repeated skips are fine
    k3, _, rej = oracle.kv_append_checked(kn, vn, skips, kc, vc)
    assert not rej
    assert np.array_equal(k3.reshape(nb * bs, hkv, d)[slots[0]], kn[0])
    assert np.array_equal(k3.reshape(nb * bs, hkv, d)[slots[1]],
                          kc.reshape(nb * bs, hkv, d)[slots[1]])


# ---------------------------------------------------------------------------
# Paging is address translation: paged == contiguous, and pages may sit
# anywhere (permutation invariance, bitwise)
# ---------------------------------------------------------------------------
def _random_contiguous(rng, lens, hkv, d):
    return [oracle.f64_to_bf16_bits(rng.standard_normal((L, hkv, d))) for L in lens]


def test_paged_equals_contiguous_bitwise():
    rng = np.random.default_rng(11)
    lens, hq, hkv, d, bs = [1, 15, 16, 17, 63], 8, 2, 16, 16
    ks = _random_contiguous(rng, lens, hkv, d)
    vs = _random_contiguous(rng, lens, hkv, d)
    q = oracle.f64_to_bf16_bits(rng.standard_normal((len(lens), hq, d)))
    need = [-(-L // bs) for L in lens]
    nb = sum(need) + 5
    ids = rng.permutation(nb)
    kc = oracle.f64_to_bf16_bits(rng.standard_normal((nb, bs, hkv, d)))
    vc = oracle.f64_to_bf16_bits(rng.standard_normal((nb, bs, hkv, d)))
    tables = np.full((len(lens), max(need)), -1, dtype=np.int32)
    cur = 0
    for s, L in enumerate(lens):
        for b in range(need[s]):
            pid = ids[cur]
            cur += 1
            tables[s, b] = pid
            rows = ks[s][b * bs:(b + 1) * bs]
            kc[pid, :rows.shape[0]] = rows
            vc[pid, :rows.shape[0]] = vs[s][b * bs:(b + 1) * bs]
    scale = 0.25
    paged = oracle.paged_decode_attention(q, kc, vc, tables, lens, scale)
    for s in range(len(lens)):
        contig = oracle.attention(q[s:s + 1], ks[s], vs[s], scale, causal=False)[0]
        assert np.array_equal(paged[s], contig)


def test_block_permutation_invariance_bitwise():
    w = wl.make_decode_workload(wl.TINY)
    kc, vc = wl.bf16_bits(w.k_cache), wl.bf16_bits(w.v_cache)
    q = wl.bf16_bits(w.q)
    tables = w.block_tables.numpy()
    lens = w.context_lens.numpy()
    base = oracle.paged_decode_attention(q, kc, vc, tables, lens, w.scale)
    rng = np.random.default_rng(5)
    perm = rng.permutation(kc.shape[0])
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    tables2 = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1)
    moved = oracle.paged_decode_attention(q, kc2, vc2, tables2, lens, w.scale)
    assert np.array_equal(base, moved)


# ---------------------------------------------------------------------------
# Closed forms
# ---------------------------------------------------------------------------
def test_one_hot_and_uniform_scores():
    rng = np.random.default_rng(2)
    L, hkv, d = 40, 2, 32
    k = rng.standard_normal((L, hkv, d))
    v = rng.standard_normal((L, hkv, d))
    j = 17
    k[j] *= 8.0                                       # one dominant key row per head
    q = np.zeros((1, 4, d))
    for h in range(4):
        q[0, h] = 50.0 * k[j, h // 2]
    out = oracle.attention(q, k, v, 1.0, causal=False)
    for h in range(4):
        np.testing.assert_allclose(out[0, h], v[j, h // 2], rtol=0, atol=1e-12)
    out0 = oracle.attention(np.zeros((1, 4, d)), k, v, 0.3, causal=False)
    for h in range(4):
        np.testing.assert_allclose(out0[0, h], v[:, h // 2].mean(axis=0), rtol=0, atol=1e-13)


def test_two_keys_logistic_closed_form():
    rng = np.random.default_rng(8)
    d = 6
    q = rng.standard_normal((1, 1, d))
    k = rng.standard_normal((2, 1, d))
    v = rng.standard_normal((2, 1, 5))                # d_v != d_k on purpose
    scale = 0.375                                     # exactly representable in fp32
    s0 = scale * float(q[0, 0] @ k[0, 0])
    s1 = scale * float(q[0, 0] @ k[1, 0])
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    expect = w0 * v[0, 0] + (1.0 - w0) * v[1, 0]
    out = oracle.attention(q, k, v, scale, causal=False)
    np.testing.assert_allclose(out[0, 0], expect, rtol=0, atol=1e-14)


def test_empty_context_is_zero():
    q = np.ones((1, 4, 8))
    k = np.zeros((0, 2, 8))
    assert np.array_equal(oracle.attention(q, k, k, 1.0, causal=False), np.zeros((1, 4, 8)))


def _check_causal_golden(attn):
    gold = _golden("causal_mask_example.json")
    tq, tk = gold["Tq"], gold["Tk"]
    kk = np.eye(tk)[:, None, :]                       # key j = e_j, so score(i, j) = q_i[j]
    vv = np.eye(tk)[:, None, :]
    q = np.array([[0.0, 0.0, math.log(2.0), 7.0],     # key 3 is masked for query 0
                  [math.log(2.0), math.log(3.0), 0.0, math.log(2.0)]])[:, None, :]
    out = attn(q, kk, vv, 1.0, True)[:, 0, :]
    return float(np.abs(out - np.array(gold["expected_out"])).max())


def test_causal_mask_hand_worked_example():
    assert _check_causal_golden(opa.attention) < 1e-15


# ---------------------------------------------------------------------------
# Library routine: torch scaled_dot_product_attention in float64 (GQA heads
# mapped by repeat-interleave; top-left causal equals bottom-right when the
# chunk is the whole context)
# ---------------------------------------------------------------------------
def _sdpa(q, k, v, scale, causal):
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]
    kt = torch.from_numpy(k).permute(1, 0, 2)[None]
    vt = torch.from_numpy(v).permute(1, 0, 2)[None]
    o = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, is_causal=causal, scale=scale, enable_gqa=True)
    return o[0].permute(1, 0, 2).numpy()


def _check_sdpa(attn):
    rng = np.random.default_rng(21)
    worst = 0.0
    for (n, L, hq, hkv, d, causal) in [(1, 37, 8, 2, 16, False), (1, 5, 4, 4, 8, False),
                                       (9, 9, 8, 2, 16, True), (12, 12, 6, 3, 8, True)]:
        q = rng.standard_normal((n, hq, d))
        k = rng.standard_normal((L, hkv, d))
        v = rng.standard_normal((L, hkv, d))
        scale = float(np.float32(1.0 / math.sqrt(d) * 1.7))
        ref = _sdpa(q, k, v, scale, causal)
        got = attn(q, k, v, scale, causal)
        worst = max(worst, float(np.abs(ref - got).max()))
    return worst


def test_attention_matches_torch_sdpa_float64():
    assert _check_sdpa(opa.attention) < 1e-12


# ---------------------------------------------------------------------------
# Online softmax, split-K merge, causal prefill vs repeated decode
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("tile", [1, 4, 16, 128])
def test_online_softmax_equals_one_shot(tile):
    rng = np.random.default_rng(tile)
    n, L, hq, hkv, d = 3, 150, 8, 2, 16
    q = rng.standard_normal((n, hq, d))
    k = rng.standard_normal((L, hkv, d)) * 3
    v = rng.standard_normal((L, hkv, d))
    for causal in (False, True):
        a = oracle.attention(q, k, v, 0.2, causal)
        b = oracle.online_softmax_attention(q, k, v, 0.2, tile, causal)
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


@pytest.mark.parametrize("part", [1, 7, 16, 64, 300])
def test_split_merge_equals_unsplit(part):
    rng = np.random.default_rng(100 + part)
    L, hq, hkv, d = 257, 8, 2, 16
    q = rng.standard_normal((1, hq, d))
    k = rng.standard_normal((L, hkv, d)) * 4
    v = rng.standard_normal((L, hkv, d))
    a = oracle.attention(q, k, v, 0.3, causal=False)[0]
    b = oracle.merge_partials(oracle.split_partials(q[0], k, v, 0.3, part))
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_causal_prefill_equals_repeated_decode():
    m = wl.make_mixed_workload(num_prefill=2, num_decode=1, chunk=21, prior_range=(0, 30),
                               shared_prefix=16, decode_cap=64)
    kc, vc = wl.bf16_bits(m.k_cache), wl.bf16_bits(m.v_cache)
    q = wl.bf16_bits(m.q_prefill)
    starts = m.q_start.numpy()
    tables = m.prefill_tables.numpy()
    lens = m.prefill_lens.numpy()
    pre = oracle.paged_prefill_attention(q, starts, kc, vc, tables, lens, True, m.scale)
    for s in range(len(lens)):
        n = starts[s + 1] - starts[s]
        for i in range(n):
            ctx = lens[s] - n + i + 1
            dec = oracle.paged_decode_attention(q[starts[s] + i][None], kc, vc, tables[s:s + 1],
                                                [ctx], m.scale)
            np.testing.assert_allclose(pre[starts[s] + i], dec[0], rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Brute-force recompute (no cache) == append through slot mapping + paged decode
# ---------------------------------------------------------------------------
def test_brute_force_recompute_equals_cached_paged_decode():
    rng = np.random.default_rng(7)
    d_model, hq, hkv, dh, steps, bs = 32, 4, 2, 8, 20, 4
    wq = rng.standard_normal((d_model, hq * dh)) / math.sqrt(d_model)
    wk = rng.standard_normal((d_model, hkv * dh)) / math.sqrt(d_model)
    wv = rng.standard_normal((d_model, hkv * dh)) / math.sqrt(d_model)
    x = rng.standard_normal((steps, d_model))
    nb = steps // bs + 3
    kc = np.zeros((nb, bs, hkv, dh), np.uint16)
    vc = np.zeros((nb, bs, hkv, dh), np.uint16)
    table = rng.permutation(nb)[: -(-steps // bs)].astype(np.int32)
    scale = 1.0 / math.sqrt(dh)
    rnd = oracle.f64_to_bf16_bits
    for t in range(steps):
        # naive: recompute K, V of the whole prefix (no cache)
        k_all = rnd((x[:t + 1] @ wk).reshape(t + 1, hkv, dh))
        v_all = rnd((x[:t + 1] @ wv).reshape(t + 1, hkv, dh))
        q_t = rnd((x[t] @ wq).reshape(1, hq, dh))
        naive = oracle.attention(q_t, k_all, v_all, scale, causal=False)[0]
        # cached: only token t's K, V, appended through its slot
        slot = int(table[t // bs]) * bs + t % bs
        kc, vc = oracle.kv_append(k_all[t:t + 1], v_all[t:t + 1], [slot], kc, vc)
        cached = oracle.paged_decode_attention(q_t, kc, vc, table[None], [t + 1], scale)[0]
        np.testing.assert_allclose(cached, naive, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Mutation tests: plausible mistakes planted in copies of the oracle's
# attention are caught by the pins above.
# ---------------------------------------------------------------------------
def _mutant(kind):
    def attn(q, k, v, scale, causal):
        n, hq, _ = q.shape
        L, hkv, _ = k.shape
        g = hq // hkv
        out = np.zeros((n, hq, v.shape[2]))
        sc = 1.0 if kind == "no_scale" else float(np.float32(scale))
        qpos = (np.arange(n) if kind == "top_left" else L - n + np.arange(n))
        for h in range(hq):
            kvh = h % hkv if kind == "gqa_modulo" else h // g
            kk, vv = (v, k) if kind == "swap_kv" else (k, v)
            s = (q[:, h, :] @ kk[:, kvh, :].T) * sc
            if causal:
                s = np.where(np.arange(L)[None, :] <= qpos[:, None], s, -np.inf)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            out[:, h, :] = p @ vv[:, kvh, :]
        return out
    return attn


@pytest.mark.parametrize("kind", ["no_scale", "gqa_modulo", "swap_kv"])
def test_sdpa_pin_catches_planted_mistakes(kind):
    assert _check_sdpa(_mutant(kind)) > 1e-3


def test_golden_mask_pin_catches_top_left_alignment():
    assert _check_causal_golden(_mutant("top_left")) > 1e-3
    assert _check_causal_golden(_mutant("none")) < 1e-15
