"""Chunked prefill over an FP8 (e4m3) cache on the GPU: the quantizing append
of the chunk tokens, then the prefill, against the oracle's attention over
the dequantized cache."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_52_gb300 import workloads as wl
from parity import assert_attention_close, remap_slots

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_52_gb300 import pagedkv
    pagedkv.get_device_error(clear=True)
    return pagedkv


NAMES = ("k_cache", "v_cache", "k_new", "v_new", "slot_mapping", "q_prefill", "q_start",
         "prefill_tables", "prefill_lens")


def _dev(w):
    for n in NAMES:
        setattr(w, n, getattr(w, n).to(DEV))
    return w


def _fp8_step_oracle(w, kc8, vc8, ks, vs, seqs):
    """Host copies of the FP8 pages the chosen sequences use (taken before the
    GPU step), renumbered, with the oracle's quantizing append of their chunk
    tokens applied.  Returns (k codes, v codes, tables, lens, q rows, q_start)."""
    lens = [int(x) for x in w.prefill_lens.cpu().tolist()]
    tables = w.prefill_tables.cpu().numpy()
    used = sorted({int(b) for s in seqs for b in tables[s, :wl.blocks_for(lens[s])]})
    remap = {b: i for i, b in enumerate(used)}
    idx = torch.tensor(used, dtype=torch.int64, device=kc8.device)
    kc, vc = kc8.index_select(0, idx).cpu().numpy(), vc8.index_select(0, idx).cpu().numpy()
    tab = np.full((len(seqs), tables.shape[1]), -1, dtype=np.int64)
    for r, s in enumerate(seqs):
        nb = wl.blocks_for(lens[s])
        tab[r, :nb] = [remap[int(b)] for b in tables[s, :nb]]
    qs = w.q_start.cpu().numpy()
    rows = np.concatenate([np.arange(qs[s], qs[s + 1]) for s in seqs]).astype(np.int64)
    sel = torch.tensor(rows, dtype=torch.int64, device=w.q_prefill.device)
    slots = remap_slots(w.slot_mapping.cpu().numpy()[rows], remap)
    kc, vc = oracle.kv_append_fp8(wl.bf16_bits(w.k_new.index_select(0, sel)),
                                  wl.bf16_bits(w.v_new.index_select(0, sel)), slots, kc, vc, ks, vs)
    q_start = np.concatenate([[0], np.cumsum([qs[s + 1] - qs[s] for s in seqs])])
    return kc, vc, tab, [lens[s] for s in seqs], rows, q_start


def _fp8_oracle(w, kc8, vc8, ks, vs, causal, seqs):
    """Oracle step (quantizing append, then prefill) of the chosen sequences."""
    kc, vc, tab, lens, rows, q_start = _fp8_step_oracle(w, kc8, vc8, ks, vs, seqs)
    sel = torch.tensor(rows, dtype=torch.int64, device=w.q_prefill.device)
    out = oracle.paged_prefill_attention_fp8(wl.bf16_bits(w.q_prefill.index_select(0, sel)),
                                             q_start, kc, vc, tab, lens, causal, w.scale, ks, vs)
    return out, rows


def _step(pk, w, kc8, vc8, ks, vs, causal, max_q_len):
    kc, vc = kc8.clone(), vc8.clone()
    pk.kv_append_fp8(w.k_new, w.v_new, w.slot_mapping, kc, vc, ks, vs)
    out = pk.paged_prefill_attention_fp8(w.q_prefill, w.q_start, kc, vc, w.prefill_tables,
                                         w.prefill_lens, causal, w.scale, ks, vs,
                                         max_q_len=max_q_len)
    torch.cuda.synchronize()
    return out, kc, vc


PRIORS = [0, 40, 17, 300, 1000, 5]
CHUNKS = [5, 130, 1, 129, 64, 16]


@pytest.mark.parametrize("hq,hkv,d", [(8, 8, 128), (16, 4, 64), (64, 8, 128), (32, 2, 64)])
@pytest.mark.parametrize("causal", [True, False])
def test_fp8_prefill_groups_and_ragged(pk, hq, hkv, d, causal):
    w = _dev(wl.make_chunked_workload(hq, hkv, d, PRIORS, CHUNKS))
    ks, vs = 0.03125, 0.03125
    kc8, vc8 = wl.fp8_pools(w, ks, vs)
    ref, _ = _fp8_oracle(w, kc8, vc8, ks, vs, causal, range(len(CHUNKS)))
    out, _, _ = _step(pk, w, kc8, vc8, ks, vs, causal, max(CHUNKS))
    assert_attention_close(out.cpu().numpy(), ref, f"fp8 prefill {hq}/{hkv} d{d} {causal}")
    assert pk.get_device_error(clear=True) == 0


def test_fp8_prefill_outlier_keys_and_unequal_scales(pk):
    # 70B-GQA heads with the x100 outlier K rows; k_scale 2, v_scale 1/32
    w = wl.make_chunked_workload(64, 8, 128, [1024, 700, 2000], [512, 64, 129])
    g = torch.Generator().manual_seed(77)
    rows = torch.randperm(w.k_cache.shape[0] * 16 * 8, generator=g)[:200]
    flat = w.k_cache.view(-1, 128)
    flat[rows] = (flat[rows].float() * 100).to(torch.bfloat16)
    w = _dev(w)
    ks, vs = wl.FP8_SCALES["gqa70b"]
    kc8, vc8 = wl.fp8_pools(w, ks, vs)
    ref, _ = _fp8_oracle(w, kc8, vc8, ks, vs, True, range(3))
    out, _, _ = _step(pk, w, kc8, vc8, ks, vs, True, 512)
    assert_attention_close(out.cpu().numpy(), ref, "fp8 prefill outliers")
    assert pk.get_device_error(clear=True) == 0


def test_fp8_prefill_nan_codes_past_the_length(pk):
    w = _dev(wl.make_chunked_workload(16, 4, 128, PRIORS, CHUNKS))
    ks, vs = 0.03125, 0.03125
    kc8, vc8 = wl.fp8_pools(w, ks, vs)
    ref, _ = _fp8_oracle(w, kc8, vc8, ks, vs, True, range(len(CHUNKS)))
    kc, vc = kc8.clone(), vc8.clone()
    pk.kv_append_fp8(w.k_new, w.v_new, w.slot_mapping, kc, vc, ks, vs)
    tables = w.prefill_tables.cpu().numpy()
    for s, L in enumerate(w.prefill_lens.cpu().tolist()):
        if L % 16:
            b = int(tables[s, (L - 1) // 16])
            kc[b, L % 16:] = 0x7F
            vc[b, L % 16:] = 0x7F
    out = pk.paged_prefill_attention_fp8(w.q_prefill, w.q_start, kc, vc, w.prefill_tables,
                                         w.prefill_lens, True, w.scale, ks, vs,
                                         max_q_len=max(CHUNKS))
    torch.cuda.synchronize()
    assert_attention_close(out.cpu().numpy(), ref, "fp8 prefill NaN tail codes")
    assert pk.get_device_error(clear=True) == 0


def test_fp8_prefill_bad_block_id_is_flagged(pk):
    w = _dev(wl.make_chunked_workload(8, 2, 64, [40, 17], [30, 1]))
    kc8, vc8 = wl.fp8_pools(w, 0.03125, 0.03125)
    tables = w.prefill_tables.clone()
    tables[0, 1] = 1 << 20
    pk.get_device_error(clear=True)
    out = pk.paged_prefill_attention_fp8(w.q_prefill, w.q_start, kc8, vc8, tables,
                                         w.prefill_lens, True, w.scale, 0.03125, 0.03125,
                                         max_q_len=30)
    torch.cuda.synchronize()
    assert pk.get_device_error(clear=True) & 0x2
    assert torch.isfinite(out).all()


def test_fp8_mixed_step_prefill_sampled(pk):
    # the full mixed step's 8 chunks (512 new tokens each, 1024-token shared
    # prefix) over FP8 pools; sampled query rows of three chunks against the
    # oracle (row i of a causal chunk of n is the FP8 decode over the first
    # context_len - n + i + 1 tokens)
    w = wl.make_mixed_workload(wl.MIXED, device=DEV, gen_device=DEV)
    ks, vs = 0.03125, 0.03125
    kc8, vc8 = wl.fp8_pools(w, ks, vs)
    seqs = [0, 3, 7]
    kc, vc, tab, lens, rows, q_start = _fp8_step_oracle(w, kc8, vc8, ks, vs, seqs)
    out, _, _ = _step(pk, w, kc8, vc8, ks, vs, True, 512)
    q = wl.bf16_bits(w.q_prefill.index_select(0, torch.tensor(rows, device=DEV)))
    got, ref = [], []
    for r in range(len(seqs)):
        n = int(q_start[r + 1] - q_start[r])
        for i in (0, 1, 17, 255, 256, n - 2, n - 1):
            row = int(q_start[r]) + i
            ref.append(oracle.paged_decode_attention_fp8(q[row][None], kc, vc, tab[r:r + 1],
                                                         [lens[r] - n + i + 1], w.scale, ks,
                                                         vs)[0])
            got.append(out[int(rows[row])].cpu().numpy())
    assert_attention_close(np.stack(got), np.stack(ref), "fp8 mixed-step prefill")
    assert pk.get_device_error(clear=True) == 0


def test_fp8_prefill_limited_sms_equals_grid(pk):
    # the persistent launch on at most N SMs computes the same tiles in the
    # same arithmetic: bitwise the grid launch's output, for any N
    w = _dev(wl.make_chunked_workload(64, 8, 128, [500, 0, 33, 2000], [300, 77, 129, 64],
                                      config_id=9))
    ks, vs = wl.FP8_SCALES["gqa70b"]
    kc8, vc8 = wl.fp8_pools(w, ks, vs)
    grid, kc, vc = _step(pk, w, kc8, vc8, ks, vs, True, 300)
    for ctas in (1, 9, 100000):
        out = pk.paged_prefill_attention_fp8(w.q_prefill, w.q_start, kc, vc, w.prefill_tables,
                                             w.prefill_lens, True, w.scale, ks, vs,
                                             max_q_len=300, max_ctas=ctas)
        torch.cuda.synchronize()
        assert torch.equal(out, grid), f"max_ctas={ctas}"
    ref, _ = _fp8_oracle(w, kc8, vc8, ks, vs, True, range(4))
    assert_attention_close(grid.cpu().numpy(), ref, "fp8 prefill (grid and limited)")
    assert pk.get_device_error(clear=True) == 0


def test_fp8_prefill_dispatch_order_many_sequences(pk):
    # the widening pass ranks the sequences (more than a warp of them, with
    # ties and empty chunks) and the prefill runs them in that order; every
    # row is computed, grid and persistent launches agree bitwise
    g = np.random.default_rng(14)
    priors = [int(x) for x in g.integers(1, 300, 70)]
    chunks = [int(x) for x in g.integers(1, 40, 70)]
    for s in (3, 4):
        priors[s], chunks[s] = 64, 16
    chunks[20] = 0
    w = _dev(wl.make_chunked_workload(16, 4, 128, priors, chunks, config_id=15))
    ks, vs = wl.FP8_SCALES["tiny"]
    kc8, vc8 = wl.fp8_pools(w, ks, vs)
    grid, kc, vc = _step(pk, w, kc8, vc8, ks, vs, True, 39)
    assert bool(torch.isfinite(grid).all())
    lim = pk.paged_prefill_attention_fp8(w.q_prefill, w.q_start, kc, vc, w.prefill_tables,
                                         w.prefill_lens, True, w.scale, ks, vs, max_q_len=39,
                                         max_ctas=23)
    torch.cuda.synchronize()
    assert torch.equal(lim, grid)
    ref, _ = _fp8_oracle(w, kc8, vc8, ks, vs, True, range(70))
    assert_attention_close(grid.cpu().numpy(), ref, "fp8 prefill, 70 sequences")
    assert pk.get_device_error(clear=True) == 0
