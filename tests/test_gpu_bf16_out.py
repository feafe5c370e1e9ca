"""The bf16-output entry points of the decode and the prefill.

Both compute in float32 as their float32 entry points do and round only in
the final store, to the nearest bf16 with ties to even.  So the checks are:

* bitwise: the bf16 output equals the float32 entry point's output rounded
  to bf16 on the CPU by torch (its conversion rounds to nearest even), on
  every path that writes the output -- the unsplit decode, the split-K merge
  in its four-wide and scalar forms, empty contexts, the prefill with and
  without its workspace;
* against the oracle: bf16 keeps 8 significant bits, so its numbers in
  [1, 2) are 2^-7 apart and rounding x to the nearest moves it by at most
  2^-8 |x| (the unit roundoff).  With |x - ref| within the float32 tolerance,
  |bf16(x) - ref| - 2^-8 |ref| <= ATOL (1 + 2^-8) element-wise, and the row
  2-norm error grows by at most 2^-8 (1 + ROW_RTOL) relative.
"""

import numpy as np
import pytest
import torch

from paged_kv_cache_52_gb300 import workloads as wl
from parity import ATOL, ROW_RTOL, DecodeStepOracle, PrefillStepOracle, attention_errors
from test_gpu_prefill import CHUNKS, PRIORS, SHAPES
from test_gpu_prefill import _to_dev as _prefill_to_dev

pytestmark = pytest.mark.gpu

DEV = "cuda"
U_BF16 = 2.0 ** -8   # unit roundoff of bf16 (8 significant bits)


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_52_gb300 import pagedkv
    pagedkv.get_device_error(clear=True)
    return pagedkv


def assert_bf16_rounding_of(got_bf16: torch.Tensor, f32: torch.Tensor, what: str):
    want = f32.cpu().to(torch.bfloat16)
    got = got_bf16.cpu()
    assert got.dtype == torch.bfloat16
    diff = (got.view(torch.int16) != want.view(torch.int16))
    assert not bool(diff.any()), f"{what}: {int(diff.sum())} values differ from the rounded float32"


def assert_bf16_close_to_oracle(got_bf16: torch.Tensor, ref: np.ndarray, what: str):
    got = got_bf16.cpu().double().numpy()
    ref = np.asarray(ref, dtype=np.float64)
    excess = np.abs(got - ref) - U_BF16 * np.abs(ref)
    assert float(excess.max(initial=0.0)) <= ATOL * (1 + U_BF16), what
    _, row_rel = attention_errors(got, ref)
    assert row_rel <= ROW_RTOL + U_BF16 * (1 + ROW_RTOL), f"{what}: row rel {row_rel:.3e}"


def _decode_dev(w):
    for name in ("q", "k_cache", "v_cache", "k_new", "v_new", "slot_mapping", "block_tables",
                 "context_lens"):
        setattr(w, name, getattr(w, name).to(DEV))
    return w


EDGE_LENS = [1, 15, 16, 17, 33, 200, 0, 161]


@pytest.mark.parametrize("hq,hkv,d", [(8, 8, 128), (8, 4, 64), (64, 8, 128), (16, 16, 64)])
@pytest.mark.parametrize("pb", [0, 1, 3])
def test_decode_bf16_out(pk, hq, hkv, d, pb):
    spec = wl.DecodeSpec("edge", 11, len(EDGE_LENS), hq, hkv, d, lens=tuple(EDGE_LENS))
    w = wl.make_decode_workload(spec, lens_override=EDGE_LENS)
    w.slot_mapping[EDGE_LENS.index(0)] = -1        # the empty sequence appends nothing
    ref = DecodeStepOracle(w, range(w.num_seqs)).output()
    w = _decode_dev(w)
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    pk.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    kw = dict(max_context_len=max(EDGE_LENS), partition_blocks=pb)
    f32 = pk.paged_decode_attention(w.q, kc, vc, w.block_tables, w.context_lens, w.scale, **kw)
    bf = pk.paged_decode_attention(w.q, kc, vc, w.block_tables, w.context_lens, w.scale,
                                   out_dtype=torch.bfloat16, **kw)
    # an output 2 bytes past an 8-byte boundary takes the merge's scalar form
    S = w.q.shape[0]
    buf = torch.full((S * hq * d + 1,), float("nan"), dtype=torch.bfloat16, device=DEV)
    shifted = buf[1:].view(S, hq, d)
    assert shifted.data_ptr() % 8 == 2
    pk.paged_decode_attention(w.q, kc, vc, w.block_tables, w.context_lens, w.scale, out=shifted,
                              **kw)
    torch.cuda.synchronize()
    tag = f"decode {hq}/{hkv} d{d} pb={pb}"
    assert_bf16_rounding_of(bf, f32, tag)
    assert_bf16_rounding_of(shifted, f32, tag + " (2-byte aligned out)")
    assert_bf16_close_to_oracle(bf, ref, tag)
    assert bool((bf[EDGE_LENS.index(0)] == 0).all())
    assert pk.get_device_error(clear=True) == 0


def test_decode_bf16_out_full_size_gqa70b(pk):
    # the 70B-GQA decode workload in the automatic split plan the benchmark times
    w = wl.make_decode_workload(wl.DECODE_SPECS["gqa70b"], device=DEV, gen_device=DEV)
    kc, vc = w.k_cache, w.v_cache
    pk.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    mcl = max(w.meta["lens"])
    f32 = pk.paged_decode_attention(w.q, kc, vc, w.block_tables, w.context_lens, w.scale,
                                    max_context_len=mcl)
    bf = pk.paged_decode_attention(w.q, kc, vc, w.block_tables, w.context_lens, w.scale,
                                   max_context_len=mcl, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert_bf16_rounding_of(bf, f32, "gqa70b")
    assert pk.get_device_error(clear=True) == 0
    del w, kc, vc
    torch.cuda.empty_cache()


def _prefill(pk, w, causal, out_dtype, workspace):
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    pk.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    ws = None
    if workspace:
        ws = pk.prefill_workspace(w.prefill_lens.shape[0], w.prefill_tables.shape[1],
                                  kc.shape[2], kc.shape[3], kc.device)
    mql = int((w.q_start[1:] - w.q_start[:-1]).max())
    out = torch.full(w.q_prefill.shape, float("nan"), dtype=out_dtype, device=DEV)
    pk.paged_prefill_attention(w.q_prefill, w.q_start, kc, vc, w.prefill_tables, w.prefill_lens,
                               causal, w.scale, out=out, max_q_len=mql, workspace=ws)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("hq,hkv,d", SHAPES)
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("workspace", [True, False])
def test_prefill_bf16_out(pk, hq, hkv, d, causal, workspace):
    w = wl.make_chunked_workload(hq, hkv, d, PRIORS, CHUNKS)
    ref = PrefillStepOracle(w, range(len(CHUNKS)), causal=causal).output()
    w = _prefill_to_dev(w)
    f32 = _prefill(pk, w, causal, torch.float32, workspace)
    bf = _prefill(pk, w, causal, torch.bfloat16, workspace)
    tag = f"prefill {hq}/{hkv} d{d} causal={causal} workspace={workspace}"
    assert_bf16_rounding_of(bf, f32, tag)
    assert_bf16_close_to_oracle(bf, ref, tag)
    assert pk.get_device_error(clear=True) == 0


def test_prefill_bf16_out_rejects_sm_limit(pk):
    w = _prefill_to_dev(wl.make_chunked_workload(8, 8, 128, [10], [20]))
    ws = pk.prefill_workspace(1, w.prefill_tables.shape[1], 8, 128, DEV)
    with pytest.raises(Exception):
        pk.paged_prefill_attention(w.q_prefill, w.q_start, w.k_cache, w.v_cache,
                                   w.prefill_tables, w.prefill_lens, True, w.scale,
                                   workspace=ws, max_ctas=16, out_dtype=torch.bfloat16)


def test_fp8_decode_bf16_out(pk):
    # FP8 pools: the same kernel arithmetic, rounded in the final store, on
    # the unsplit path and through the merge (both merge forms)
    lens = [1, 16, 17, 200, 0, 900, 33]
    spec = wl.DecodeSpec("fp8edge", 12, len(lens), 64, 8, 128, lens=tuple(lens))
    w = _decode_dev(wl.make_decode_workload(spec, lens_override=lens))
    ks, vs = wl.FP8_SCALES["tiny"]
    kc8, vc8 = wl.fp8_pools(w, ks, vs)
    for pb in (0, 2):
        kw = dict(max_context_len=max(lens), partition_blocks=pb)
        f32 = pk.paged_decode_attention_fp8(w.q, kc8, vc8, w.block_tables, w.context_lens,
                                            w.scale, ks, vs, **kw)
        bf = pk.paged_decode_attention_fp8(w.q, kc8, vc8, w.block_tables, w.context_lens,
                                           w.scale, ks, vs, out_dtype=torch.bfloat16, **kw)
        S, hq, d = w.q.shape
        buf = torch.zeros(S * hq * d + 1, dtype=torch.bfloat16, device=DEV)
        shifted = buf[1:].view(S, hq, d)
        pk.paged_decode_attention_fp8(w.q, kc8, vc8, w.block_tables, w.context_lens, w.scale,
                                      ks, vs, out=shifted, **kw)
        torch.cuda.synchronize()
        assert_bf16_rounding_of(bf, f32, f"fp8 decode pb={pb}")
        assert_bf16_rounding_of(shifted, f32, f"fp8 decode pb={pb}, 2-byte aligned out")
    assert pk.get_device_error(clear=True) == 0


@pytest.mark.parametrize("K,pb", [(2, 0), (4, 2), (3, 0)])
def test_verify_bf16_out(pk, K, pb):
    lens = [4, 17, 33, 300, 1000, 16, 250, 129]
    w = wl.make_chunked_workload(64, 8, 128, [L - K for L in lens], [K] * len(lens),
                                 config_id=8)
    w = _prefill_to_dev(w)
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    pk.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    S = len(lens)
    q = w.q_prefill.view(S, K, 64, 128)
    kw = dict(max_context_len=max(lens), partition_blocks=pb)
    f32 = pk.paged_verify_attention(q, kc, vc, w.prefill_tables, w.prefill_lens, w.scale, **kw)
    bf = pk.paged_verify_attention(q, kc, vc, w.prefill_tables, w.prefill_lens, w.scale,
                                   out_dtype=torch.bfloat16, **kw)
    torch.cuda.synchronize()
    assert_bf16_rounding_of(bf, f32, f"verify K={K} pb={pb}")
    assert pk.get_device_error(clear=True) == 0
