"""The prefill with a workspace (V pages converted to f16, P as one f16
operand in the P V product) against the CPU oracle: the same cases as the
bf16 hi + lo prefill, plus rows past the length holding NaN and a V value
beyond f16's range."""

import numpy as np
import pytest
import torch

from paged_kv_cache_52_gb300 import workloads as wl
from parity import PrefillStepOracle, assert_attention_close, attention_errors
from test_gpu_prefill import CHUNKS, PRIORS, SHAPES, _to_dev, mixed_prefill_tiles_close

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_52_gb300 import pagedkv
    pagedkv.get_device_error(clear=True)
    return pagedkv


def run_f16pv(pk, w, causal=True, max_q_len=None, poison=False):
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    pk.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    if poison:  # rows past each length in its last page hold NaN
        tables = w.prefill_tables.cpu().numpy()
        for s, L in enumerate(w.prefill_lens.cpu().tolist()):
            if L % 16:
                b = int(tables[s, (L - 1) // 16])
                kc[b, L % 16:] = float("nan")
                vc[b, L % 16:] = float("nan")
    S = w.prefill_lens.shape[0]
    ws = pk.prefill_workspace(S, w.prefill_tables.shape[1], kc.shape[2], kc.shape[3], kc.device)
    mql = max_q_len or int((w.q_start[1:] - w.q_start[:-1]).max())
    out = torch.full(w.q_prefill.shape, float("nan"), dtype=torch.float32, device=DEV)
    pk.paged_prefill_attention(w.q_prefill, w.q_start, kc, vc, w.prefill_tables, w.prefill_lens,
                               causal, w.scale, out=out, max_q_len=mql, workspace=ws)
    torch.cuda.synchronize()
    return out, kc, vc


@pytest.mark.parametrize("hq,hkv,d", SHAPES)
@pytest.mark.parametrize("causal", [True, False])
def test_f16pv_groups_and_ragged_lengths(pk, hq, hkv, d, causal):
    w = wl.make_chunked_workload(hq, hkv, d, PRIORS, CHUNKS)
    ref = PrefillStepOracle(w, range(len(CHUNKS)), causal=causal).output()
    out, _, _ = run_f16pv(pk, _to_dev(w), causal)
    assert_attention_close(out.cpu().numpy(), ref, f"f16 PV {hq}/{hkv} d{d} causal={causal}")
    assert pk.get_device_error(clear=True) == 0


def test_f16pv_long_chunks_and_outlier_keys(pk):
    w = wl.make_chunked_workload(64, 8, 128, [4000, 700, 900], [300, 513, 200], config_id=7)
    g = torch.Generator().manual_seed(5)
    kc = w.k_cache.float()
    rows = torch.randperm(kc.shape[0] * 16, generator=g)[:60]
    kc.view(-1, 8, 128)[rows] *= 100.0
    w.k_cache = kc.to(torch.bfloat16)
    ref = PrefillStepOracle(w, [0, 1, 2]).output()
    out, _, _ = run_f16pv(pk, _to_dev(w))
    max_abs, _ = assert_attention_close(out.cpu().numpy(), ref, "f16 PV long + outliers")
    assert max_abs < 1e-3   # 2^-11 relative in P, measured well inside the bound
    assert pk.get_device_error(clear=True) == 0


def test_f16pv_nan_rows_past_the_length(pk):
    w = wl.make_chunked_workload(16, 4, 128, PRIORS, CHUNKS)
    ref = PrefillStepOracle(w, range(len(CHUNKS))).output()
    out, _, _ = run_f16pv(pk, _to_dev(w), poison=True)
    assert_attention_close(out.cpu().numpy(), ref, "f16 PV NaN tails")
    assert pk.get_device_error(clear=True) == 0


def test_f16pv_value_beyond_f16_range_is_flagged(pk):
    w = wl.make_chunked_workload(8, 2, 64, [40], [8], config_id=15)
    w.v_cache.view(-1)[0:4] = 1e6          # in some page; out of f16's range
    w = _to_dev(w)
    pk.get_device_error(clear=True)
    tables = w.prefill_tables.clone()
    tables[0, 0] = 0                       # make sure block 0 is read
    w.prefill_tables = tables
    run_f16pv(pk, w)
    assert pk.get_device_error(clear=True) & 0x40


def test_f16pv_full_mixed_step(pk):
    w = wl.make_mixed_workload(device=DEV, gen_device=DEV)
    out, _, _ = run_f16pv(pk, w, max_q_len=512)
    assert torch.isfinite(out).all()
    mixed_prefill_tiles_close(out, w, "mixed prefill (f16 P V)")
    assert pk.get_device_error(clear=True) == 0


def test_f16pv_agrees_with_hi_lo_path(pk):
    # both paths approximate the same float64 result; they differ only in P's
    # rounding, by far less than the tolerance
    w = _to_dev(wl.make_chunked_workload(64, 8, 128, [500, 0, 33], [300, 77, 129], config_id=9))
    a, kc, vc = run_f16pv(pk, w)
    b = pk.paged_prefill_attention(w.q_prefill, w.q_start, kc, vc, w.prefill_tables,
                                   w.prefill_lens, True, w.scale, max_q_len=300)
    torch.cuda.synchronize()
    max_abs, _ = attention_errors(a.cpu().numpy(), b.cpu().numpy())
    assert max_abs < 1e-3


def _limited(pk, w, kc, vc, max_ctas, causal=True, stream=None):
    S = w.prefill_lens.shape[0]
    ws = pk.prefill_workspace(S, w.prefill_tables.shape[1], kc.shape[2], kc.shape[3], kc.device)
    mql = int((w.q_start[1:] - w.q_start[:-1]).max())
    out = torch.full(w.q_prefill.shape, float("nan"), dtype=torch.float32, device=DEV)
    with torch.cuda.stream(stream or torch.cuda.current_stream()):
        pk.paged_prefill_attention(w.q_prefill, w.q_start, kc, vc, w.prefill_tables,
                                   w.prefill_lens, causal, w.scale, out=out, max_q_len=mql,
                                   workspace=ws, max_ctas=max_ctas)
    return out


@pytest.mark.parametrize("causal", [True, False])
def test_limited_sms_equals_grid_launch(pk, causal):
    # the persistent launch computes the same tiles in the same arithmetic,
    # so its output is bitwise the grid launch's, for any number of CTAs
    # (1: one CTA walks every item; more CTAs than items: the surplus exits)
    w = _to_dev(wl.make_chunked_workload(64, 8, 128, [500, 0, 33, 2000], [300, 77, 129, 64],
                                         config_id=9))
    ref_out, kc, vc = run_f16pv(pk, w, causal)
    for ctas in (1, 7, 148, 100000):
        out = _limited(pk, w, kc, vc, ctas, causal)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out), f"max_ctas={ctas}"
    ref = PrefillStepOracle(w, range(4), causal=causal).output()
    assert_attention_close(ref_out.cpu().numpy(), ref, "limited prefill vs oracle")
    assert pk.get_device_error(clear=True) == 0


def test_limited_prefill_beside_decode_on_another_stream(pk):
    # the continuous-batching step with the SMs split: the prefill on at most
    # 100 SMs, the decode launched right after it on a second stream; both
    # results equal the ones computed one after the other
    w = wl.make_mixed_workload(device=DEV, gen_device=DEV, num_decode=64)
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    pk.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    dl = w.meta["decode_lens"]
    hq, d, hkv = w.q_decode.shape[1], w.q_decode.shape[2], kc.shape[2]
    dws = pk.decode_workspace(len(dl), hq, hkv, d, max(dl), kc.device)

    def decode(stream):
        with torch.cuda.stream(stream):
            return pk.paged_decode_attention(w.q_decode, kc, vc, w.decode_tables, w.decode_lens,
                                             w.scale, max_context_len=max(dl), workspace=dws)
    main = torch.cuda.current_stream()
    p_serial = _limited(pk, w, kc, vc, 148)
    d_serial = decode(main)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(main)
    p_conc = _limited(pk, w, kc, vc, 100)
    d_conc = decode(side)
    main.wait_stream(side)
    torch.cuda.synchronize()
    assert torch.equal(p_conc, p_serial)
    assert torch.equal(d_conc, d_serial)
    pre = PrefillStepOracle(w, [0, 7])
    picks = [(0, 0), (0, 511), (1, 255), (1, 511)]
    qs = w.q_start.cpu().numpy()
    got = np.stack([p_conc[int(qs[[0, 7][si]]) + i].cpu().numpy() for si, i in picks])
    assert_attention_close(got, pre.rows_output(picks), "limited prefill beside decode")
    assert pk.get_device_error(clear=True) == 0


def _many_sequences(seed, n=70):
    # more sequences than a warp, with tied context lengths and empty chunks
    g = np.random.default_rng(seed)
    priors = [int(x) for x in g.integers(1, 300, n)]
    chunks = [int(x) for x in g.integers(1, 40, n)]
    for s in (5, 6, 7):                     # three sequences of equal length
        priors[s], chunks[s] = 100, 20
    chunks[10] = chunks[11] = 0             # nothing to compute for these
    return priors, chunks


def test_dispatch_order_covers_every_sequence_once(pk):
    # the page pass ranks the sequences by context length and the prefill
    # runs them in that order: every sequence is still computed (no output
    # row left NaN), the result matches the oracle, and the persistent
    # launch, which takes the same order from its counter, agrees bitwise
    priors, chunks = _many_sequences(12)
    w = _to_dev(wl.make_chunked_workload(16, 4, 64, priors, chunks, config_id=13))
    out, kc, vc = run_f16pv(pk, w)
    assert bool(torch.isfinite(out).all())
    for ctas in (1, 37):
        lim = _limited(pk, w, kc, vc, ctas)
        torch.cuda.synchronize()
        assert torch.equal(lim, out), f"max_ctas={ctas}"
    ref = PrefillStepOracle(w, range(len(chunks))).output()
    assert_attention_close(out.cpu().numpy(), ref, "70 sequences, dispatch order")
    assert pk.get_device_error(clear=True) == 0
