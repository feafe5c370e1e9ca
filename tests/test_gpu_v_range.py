"""How the accuracy of the paths that feed P to the P V product as one f16
operand depends on the size of V.

f16 rounds each weight p_j with a relative error of at most 2^-11, and the
row sum adds the weights as rounded, so the output is a convex combination of
V rows whose weights are off by at most 2^-11 relative: the error of an output
element is at most 2^-11 * max_j |v_j - out| <= 2^-10 * max|V|.  The bound
scales with V while the parity tolerance's 2e-3 is absolute, so these tests scale V
by 1, 8, 32 and 128 (exact powers of two in bf16), check the derived bound
and the 1e-2 row-wise relative bound, and print the absolute error of each
case (``pytest -s``) to record where it leaves 2e-3.  The plain prefill entry
point (P as bf16 hi + lo, ~2^-17 relative) is checked beside it to stay far
below that: its accuracy does not hinge on |V|.
"""

import numpy as np
import pytest
import torch

from paged_kv_cache_52_gb300 import workloads as wl
from parity import PrefillStepOracle, attention_errors, ROW_RTOL
from test_gpu_fp8 import _fp8_oracle, _step as fp8_step, _dev as fp8_dev
from test_gpu_prefill import run_prefill, _to_dev
from test_gpu_prefill_f16pv import run_f16pv

pytestmark = pytest.mark.gpu

DEV = "cuda"
SCALES = [1, 8, 32, 128]
F16_P_BOUND = 2.0 ** -10    # times max|V|: f16 rounding of P (2^-11) times |v - out| <= 2 max|V|
HI_LO_BOUND = 2.0 ** -14    # times max|V|: bf16 hi + lo P (2^-17), with room for fp32 sums


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_52_gb300 import pagedkv
    pagedkv.get_device_error(clear=True)
    return pagedkv


def _scale_v(w, s):
    """V pools and new V rows times s (a power of two: exact in bf16)."""
    w.v_cache = (w.v_cache.float() * s).to(torch.bfloat16)
    w.v_new = (w.v_new.float() * s).to(torch.bfloat16)
    return w


# rows that see few keys (prior 0) weigh few V rows: the largest P-rounding error
PRIORS = [0, 40, 300, 1000]
CHUNKS = [130, 64, 129, 16]


@pytest.mark.parametrize("s", SCALES)
def test_prefill_f16_p_error_scales_with_max_v(pk, s):
    w = _scale_v(wl.make_chunked_workload(64, 8, 128, PRIORS, CHUNKS, config_id=12), s)
    ref = PrefillStepOracle(w, range(len(CHUNKS))).output()
    vmax = float(max(w.v_cache.float().abs().max(), w.v_new.float().abs().max()))
    w = _to_dev(w)
    f16, _, _ = run_f16pv(pk, w)
    plain, _, _ = run_prefill(pk, w)
    e16, r16 = attention_errors(f16.cpu().numpy(), ref)
    epl, rpl = attention_errors(plain.cpu().numpy(), ref)
    print(f"\nprefill V x{s}: max|V| {vmax:.1f}; f16 P (workspace) max|err| {e16:.3e} "
          f"({e16 / vmax:.2e} of max|V|), row rel {r16:.2e}; bf16 hi+lo (plain) max|err| "
          f"{epl:.3e}, row rel {rpl:.2e}")
    assert e16 <= F16_P_BOUND * vmax and r16 <= ROW_RTOL
    assert epl <= HI_LO_BOUND * vmax and rpl <= ROW_RTOL
    assert pk.get_device_error(clear=True) == 0


@pytest.mark.parametrize("s", SCALES)
def test_fp8_decode_f16_p_error_scales_with_max_v(pk, s):
    w = fp8_dev(wl.make_decode_workload(wl.GQA_70B, lens_override=[1024, 3000, 777, 17, 2049]))
    ks, vs0 = wl.FP8_SCALES["gqa70b"]
    kc8, vc8 = wl.fp8_pools(w, ks, vs0)
    vs = vs0 * s                                  # the dequantized V scales by s
    ref = _fp8_oracle(w, kc8, vc8, ks, vs, range(5))
    out, _, vc = fp8_step(pk, w, kc8, vc8, ks, vs)
    codes = vc.view(torch.float8_e4m3fn).float().abs()
    vmax = float(codes.max()) * vs
    err, rel = attention_errors(out.cpu().numpy(), ref)
    print(f"\nFP8 decode V x{s}: max|V| {vmax:.1f}; max|err| {err:.3e} "
          f"({err / vmax:.2e} of max|V|), row rel {rel:.2e}")
    assert np.isfinite(out.cpu().numpy()).all()
    assert err <= F16_P_BOUND * vmax and rel <= ROW_RTOL
    assert pk.get_device_error(clear=True) == 0
