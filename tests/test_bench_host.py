"""Host logic of bench.py on the CPU: the compact per-config digest printed
at the end of the JSON line carries every workload's headline numbers."""

import json

import bench


def test_per_config_summary_carries_every_workload():
    line = {
        "value": 6900.0, "roofline": {"frac": 1.01}, "decode_tokens_per_s": 370000.0,
        "decode_tokens_per_s_80_layers_attention_only": 4625.0,
        "cpu_baseline": {"value": 0.9},
        "other_decode_workloads": {
            "mha7b": {"decode_GBps": 7100.0, "decode_frac_of_hbm": 1.05,
                      "decode_tokens_per_s": 1.0, "cpu_baseline": {"value": 1.1}},
            "long128k": {"decode_GBps": 6700.0, "decode_frac_of_hbm": 0.99,
                         "decode_tokens_per_s": 2.0, "cpu_baseline": None}},
        "fp8_cache": {"decode_GBps": 6400.0, "decode_frac_of_hbm": 0.94},
        "mixed_step": {"ms_per_step": 1.05, "roofline_step_ms": 0.77,
                       "prefill": {"frac": 0.57, "plain_entry_point_frac": 0.44},
                       "decode": {"unique_GBps": 5800.0},
                       "two_streams_sm_split": {"ms_per_step": 0.91},
                       "unified": {"ms_per_step": 0.89}, "cpu_baseline": {"value": 17000.0}},
        "small_batch_decode": {"8": {"eager_us": 40.0, "graph_us": 41.0}},
    }
    out = bench.per_config_summary(line, 6785.9)
    assert set(out) == {"peak_GBps", "gqa70b", "mha7b", "long128k", "gqa70b_fp8", "mixed",
                        "small_batch_us"}
    assert out["gqa70b"]["cpu_GBps"] == 0.9 and out["mha7b"]["cpu_GBps"] == 1.1
    assert out["long128k"]["cpu_GBps"] is None
    assert out["mixed"]["fused_ms"] == 0.89 and out["mixed"]["cpu_ms"] == 17000.0
    # short enough to stay in the last 1500 characters of the line with the
    # CPU baseline before it
    assert len(json.dumps(out)) < 1100


def test_prefill_flops_count_the_visible_keys():
    # a causal chunk of n tokens after p cached ones: query i sees p + i + 1
    # keys, so n p + n (n + 1) / 2 (query, key) pairs; brute force on small
    # ragged cases, then the mixed step's 8 chunks x 64 heads x d 128 x 4
    # flops per pair, the figure the bench's prefill rows divide by
    import dataclasses

    from paged_kv_cache_52_gb300 import workloads as wl
    for priors, chunks in (([0], [1]), ([5, 0, 17], [3, 9, 1]), ([40], [64])):
        brute = sum(p + i + 1 for p, n in zip(priors, chunks) for i in range(n))
        assert bench.prefill_flops([p + n for p, n in zip(priors, chunks)], chunks) == brute
    priors = wl.mixed_prefill_priors()
    assert 4 * 128 * 64 * bench.prefill_flops([p + 512 for p in priors], [512] * 8) == \
        518_533_414_912
    # the priors are the mixed workload's own draw (a small spec of the same
    # recipe, so the pools stay small)
    spec = dataclasses.replace(wl.MIXED, num_prefill=3, num_decode=2, chunk=32,
                               prior_range=(0, 64), shared_prefix=16, max_len=256,
                               decode_median=64.0)
    w = wl.make_mixed_workload(spec)
    assert wl.mixed_prefill_priors(spec) == [L - 32 for L in w.meta["prefill_lens"]]
