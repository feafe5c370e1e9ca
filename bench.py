"""Benchmark: one decode step of paged attention on the 70B-GQA layer workload.

A step is the decode hot path over one batch: KV append of the new token of
all 256 sequences, then paged decode attention (split-K + log-sum-exp merge)
over their histories (context lengths uniform in [1024, 8192], 64 query / 8
KV heads, d_head 128, 16-token blocks, bf16 with 0.1% of K rows x100).

Metric: KV GB/s (logical K+V bytes the decode reads, per second), with decode
tokens/s and the fraction of the measured HBM peak.  Inputs (~4.8 GB of KV)
are larger than L2, so no flush is needed between steps.

``python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]``
prints one JSON line.  With N > 1 (torchrun, one rank per GPU) every rank runs
its own replica of the workload (the path has no cross-GPU exchange) and the
value is the total over ranks divided by the slowest rank's time.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import resource
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from paged_kv_cache_52_gb300 import workloads as wl  # noqa: E402

METRIC = "paged decode attn: KV GB/s & % of GB300 HBM peak; decode tokens/s at 70B-GQA"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gqa70b", choices=sorted(wl.DECODE_SPECS))
    ap.add_argument("--partition-blocks", type=int, default=0)
    ap.add_argument("--separate-step", action="store_true",
                    help="time the step as two calls (kv_append, then the decode) instead of "
                         "pkv_paged_decode_step")
    ap.add_argument("--num-seqs", type=int, default=0,
                    help="shrink the workload to this many sequences (profiling runs)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="wall-time budget of the CPU oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-mixed", action="store_true",
                    help="skip the continuous-batching mixed-step measurement")
    ap.add_argument("--mixed-steps", type=int, default=30)
    ap.add_argument("--mixed-span-sweep", action="store_true",
                    help="also time the fused mixed step over a range of work-list interleaves")
    ap.add_argument("--config-cpu-seconds", type=float, default=8.0,
                    help="wall-time budget of the CPU oracle sample of each other config "
                         "(7B-MHA, 128K) and of the mixed step; 0 skips them")
    ap.add_argument("--only-verify", action="store_true",
                    help="run only the speculative-verification comparison")
    ap.add_argument("--verify-seqs", type=int, default=256,
                    help="sequences of the speculative-verification workload")
    ap.add_argument("--mixed-decodes", type=int, default=None,
                    help="shrink the mixed step to this many decode sequences (profiling runs)")
    ap.add_argument("--only-mixed", action="store_true",
                    help="time only the mixed step (profiling runs)")
    ap.add_argument("--only-fused", action="store_true",
                    help="time only the fused mixed step (append + one persistent launch), "
                         "with the decodes' shared prefix as a prefix group (profiling runs)")
    ap.add_argument("--only-append", action="store_true",
                    help="run only the bulk append probe (profiling runs)")
    ap.add_argument("--append-tokens", type=int, default=262144,
                    help="tokens of the bulk append probe")
    ap.add_argument("--append-steps", type=int, default=20)
    ap.add_argument("--only-prefill-lengths", action="store_true",
                    help="run only the prefill over chunks of 512 tokens with 1K to 32K "
                         "cached tokens before them (the rate against the length of a "
                         "CTA's work; profiling runs)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(ms: float, device) -> float:
    """The slowest rank's time (a control all-reduce; the data path has none)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbps(bytes_per_rank_step: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: every rank's bytes over the slowest rank's time."""
    return world * bytes_per_rank_step * steps / (max_ms / 1e3) / 1e9


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def workload_config(w, spec, plan):
    lens = w.meta["lens"]
    return {
        "workload": spec.name if w.num_seqs == spec.num_seqs else
        f"{spec.name}, shrunk to {w.num_seqs} sequences",
        "num_seqs": w.num_seqs, "q_heads": w.q_heads, "kv_heads": w.kv_heads,
        "d_head": w.d_head, "block_size": wl.BLOCK_SIZE,
        "context_len_min": min(lens), "context_len_max": max(lens),
        "context_len_mean": round(sum(lens) / len(lens), 1),
        "kv_bytes_per_step": w.kv_bytes(),
        "partition_blocks": plan[0], "num_parts": plan[1],
        "l2": "inputs larger than L2 (KV per step >> 129 MB); no flush",
        "step": "kv_append(1 token/seq) + paged_decode_attention (split-K + LSE merge), "
                "through pkv_paged_decode_step (the append's kernel runs beside the split "
                "kernel; only each sequence's last page waits for it)",
    }


class ClockSampler:
    """nvidia-smi clock/throttle samples (every 100 ms) while the GPU runs the
    step under load: a 0.6 s lead-in of the same steps, then the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def _host_sequence(w, s):
    """Host copy of what the oracle needs for sequence s of a device workload:
    its physical blocks renumbered 0..n-1 (pages may sit anywhere), its new
    token's slot in that numbering, q and the new K/V rows."""
    nb = wl.blocks_for(int(w.meta["lens"][s]))
    ids = w.block_tables[s, :nb].to(torch.int64)
    kc = wl.bf16_bits(w.k_cache.index_select(0, ids))
    vc = wl.bf16_bits(w.v_cache.index_select(0, ids))
    slot = int(w.slot_mapping[s])
    phys = ids.cpu().tolist()
    local = phys.index(slot // wl.BLOCK_SIZE) * wl.BLOCK_SIZE + slot % wl.BLOCK_SIZE
    return dict(kc=kc, vc=vc, table=[list(range(nb))], slot=[local], len=[w.meta["lens"][s]],
                q=wl.bf16_bits(w.q[s:s + 1]), k_new=wl.bf16_bits(w.k_new[s:s + 1]),
                v_new=wl.bf16_bits(w.v_new[s:s + 1]))


def cpu_oracle_sample(w, budget_s: float, seqs=None):
    """Time the CPU oracle, as it stands, on whole sequences of the workload
    (append, then decode) until the wall-time budget is spent.  Returns the
    same metric (KV GB/s) and a description; `cores` is CPU time / wall time
    of the oracle calls, i.e. the threads it actually kept busy.  `seqs`:
    the sequences to take, in order (default: all, from the first)."""
    import oracle  # CPU baseline only

    row_bytes = 2 * w.kv_heads * w.d_head * 2
    done_bytes, wall, cpu, nseq = 0, 0.0, 0.0, 0
    order = list(range(w.num_seqs)) if seqs is None else list(seqs)
    for s in order:
        if wall >= budget_s:
            break
        h = _host_sequence(w, s)
        c0, t0 = time.process_time(), time.perf_counter()
        kc, vc = oracle.kv_append(h["k_new"], h["v_new"], h["slot"], h["kc"], h["vc"])
        oracle.paged_decode_attention(h["q"], kc, vc, h["table"], h["len"], w.scale)
        wall += time.perf_counter() - t0
        cpu += time.process_time() - c0
        done_bytes += h["len"][0] * row_bytes
        nseq += 1
    value = done_bytes / wall / 1e9 if wall > 0 else None
    cores = max(1, round(cpu / wall)) if wall > 0 else 1
    info = {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
            "host_cpus": len(os.sched_getaffinity(0)),
            "sample": f"append+decode of {nseq} of {w.num_seqs} sequences "
                      f"({done_bytes / 1e9:.3f} GB of KV) in {wall:.1f} s, numpy float64"}
    return value, info


def cpu_prefill_sample(w, seqs, tiles, budget_s: float):
    """Time the CPU oracle on query tiles of prefill chunks of a mixed
    workload: the sequence's pages and its chunk's new rows to the host, the
    oracle's append, then the oracle's causal attention of query tokens
    [a, b) over the first context_len - n + b keys (those tokens are the last
    b - a positions there).  Returns (GFLOP/s, wall s, flops) with the same
    flop count as the GPU figure (4 d Hq per visible key per query row)."""
    import oracle  # CPU baseline only

    chunk = w.meta["chunk"]
    qs = w.q_start.cpu().tolist()
    hq, d = w.q_prefill.shape[1], w.q_prefill.shape[2]
    flops, wall = 0, 0.0
    for s in seqs:
        L = int(w.meta["prefill_lens"][s])
        nb = wl.blocks_for(L)
        ids = w.prefill_tables[s, :nb].to(torch.int64)
        kc = wl.bf16_bits(w.k_cache.index_select(0, ids))
        vc = wl.bf16_bits(w.v_cache.index_select(0, ids))
        rows = torch.arange(qs[s], qs[s + 1], device=w.q_prefill.device)
        phys = ids.cpu().tolist()
        slots = [phys.index(int(x) // wl.BLOCK_SIZE) * wl.BLOCK_SIZE + int(x) % wl.BLOCK_SIZE
                 for x in w.slot_mapping[qs[s]:qs[s + 1]].cpu().tolist()]
        kn = wl.bf16_bits(w.k_new.index_select(0, rows))
        vn = wl.bf16_bits(w.v_new.index_select(0, rows))
        q = wl.bf16_bits(w.q_prefill.index_select(0, rows))
        t0 = time.perf_counter()
        kc2, vc2 = oracle.kv_append(kn, vn, slots, kc, vc)
        table = list(range(nb))
        for a, b in tiles:
            ctx = L - chunk + b
            kk = oracle.gather_sequence_kv(kc2, table, ctx)
            vv = oracle.gather_sequence_kv(vc2, table, ctx)
            oracle.attention(q[a:b], kk, vv, w.scale, causal=True)
            flops += 4 * d * hq * sum(L - chunk + i + 1 for i in range(a, b))
        wall += time.perf_counter() - t0
        if wall >= budget_s:
            break
    return flops / wall / 1e9, wall, flops


def read_traffic(kernel_tag: str):
    """DRAM bytes per launch from a committed ncu summary, or None when the
    kernel source changed since the counters were taken.  The summary holds a
    line `traffic <tag> source_sha256=<hex> dram_bytes_per_launch=<int>`."""
    import hashlib

    h = hashlib.sha256()
    for f in ("paged_decode.cu", "pkv_decode_body.cuh", "pkv_device.cuh", "pkv_decode_common.cuh"):
        with open(os.path.join(ROOT, "paged_kv_cache_52_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    sha = h.hexdigest()
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None, sha
    for name in sorted(os.listdir(pdir)):
        if not name.endswith((".txt", ".md")):
            continue
        with open(os.path.join(pdir, name)) as fh:
            for ln in fh:
                parts = ln.split()
                if len(parts) >= 4 and parts[0] == "traffic" and parts[1] == kernel_tag:
                    kv = dict(p.split("=", 1) for p in parts[2:] if "=" in p)
                    if kv.get("source_sha256") == sha:
                        return int(kv["dram_bytes_per_launch"]), sha
    return None, sha


def prefill_flops(prefill_lens, chunks) -> int:
    """Algorithmic FLOPs of causal chunked prefill: QK^T and PV, 2 flops per
    multiply-add, over the keys each query sees (n * prior + n (n + 1) / 2 per
    chunk), times heads and head size.  Masked work the kernel skips or
    wastes is not counted."""
    total = 0
    for L, n in zip(prefill_lens, chunks):
        prior = L - n
        total += n * prior + n * (n + 1) // 2
    return total


def run_mixed(args, dev, pagedkv, E):
    """The continuous-batching step at full size: append 8 x 512 + 248 new
    tokens, prefill the 8 chunks (tcgen05), decode the 248 sequences."""
    w = wl.make_mixed_workload(device=dev, gen_device=dev, num_decode=args.mixed_decodes)
    kc, vc = w.k_cache, w.v_cache
    chunk = w.meta["chunk"]
    plens, dlens = w.meta["prefill_lens"], w.meta["decode_lens"]
    hq, d, hkv = w.q_prefill.shape[1], w.q_prefill.shape[2], kc.shape[2]
    max_d = max(dlens)
    ws = pagedkv.decode_workspace(len(dlens), hq, hkv, d, max_d, dev)
    pout = torch.empty(w.q_prefill.shape, dtype=torch.float32, device=dev)
    dout = torch.empty(w.q_decode.shape, dtype=torch.float32, device=dev)

    def append():
        pagedkv.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)

    pws = pagedkv.prefill_workspace(len(plens), w.prefill_tables.shape[1], hkv, d, dev)

    def prefill(max_ctas=None):
        # the workspace path: V pages to f16 first, P as one f16 operand;
        # max_ctas: a persistent launch on at most that many SMs
        pagedkv.paged_prefill_attention(w.q_prefill, w.q_start, kc, vc, w.prefill_tables,
                                        w.prefill_lens, True, w.scale, out=pout,
                                        max_q_len=chunk, workspace=pws, max_ctas=max_ctas)

    def prefill_plain():
        pagedkv.paged_prefill_attention(w.q_prefill, w.q_start, kc, vc, w.prefill_tables,
                                        w.prefill_lens, True, w.scale, out=pout,
                                        max_q_len=chunk)

    def decode():
        pagedkv.paged_decode_attention(w.q_decode, kc, vc, w.decode_tables, w.decode_lens,
                                       w.scale, out=dout, max_context_len=max_d, workspace=ws)

    for _ in range(max(3, args.warmup)):
        append(), prefill(), decode()
    torch.cuda.synchronize()
    K = args.mixed_steps
    marks = [tuple(E(enable_timing=True) for _ in range(4)) for _ in range(K)]
    for a, b, c, e in marks:
        a.record()
        append()
        b.record()
        prefill()
        c.record()
        decode()
        e.record()
    torch.cuda.synchronize()
    ms = lambda i, j: sum(m[i].elapsed_time(m[j]) for m in marks) / K  # noqa: E731
    t_step, t_app, t_pre, t_dec = ms(0, 3), ms(0, 1), ms(1, 2), ms(2, 3)
    # the plain entry point (no workspace: bf16 V, P as bf16 hi + lo)
    for _ in range(3):
        prefill_plain()
    torch.cuda.synchronize()
    c0, c1 = E(enable_timing=True), E(enable_timing=True)
    c0.record()
    for _ in range(K):
        prefill_plain()
    c1.record()
    torch.cuda.synchronize()
    t_pre_plain = c0.elapsed_time(c1) / K
    # the same decodes through the shared-prefix (cascade) path
    pblocks = w.meta["shared_prefix"] // wl.BLOCK_SIZE
    cws = torch.empty(max(1, pagedkv.lib.pkv_decode_shared_prefix_workspace_bytes(
        len(dlens), hq, hkv, d, max_d, pblocks)), dtype=torch.uint8, device=dev)

    def decode_cascade():
        pagedkv.paged_decode_attention_shared_prefix(w.q_decode, kc, vc, w.decode_tables,
                                                     w.decode_lens, w.scale, pblocks, max_d,
                                                     out=dout, workspace=cws)

    for _ in range(3):
        decode_cascade()
    torch.cuda.synchronize()
    c0, c1 = E(enable_timing=True), E(enable_timing=True)
    c0.record()
    for _ in range(K):
        decode_cascade()
    c1.record()
    torch.cuda.synchronize()
    t_casc = c0.elapsed_time(c1) / K
    # prefill and decode are independent after the append: run them on two
    # streams (the prefill is tensor-bound, the decode HBM-bound)
    main = torch.cuda.current_stream()
    s_pre, s_dec = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    # With the SMs split, the prefill runs persistent on at most `ctas` SMs
    # from a high-priority stream and the decode fills the other SMs at the
    # same time, instead of waiting for prefill CTAs that each hold a whole SM.
    s_pre_hi = torch.cuda.Stream(device=dev, priority=-1)

    def concurrent_step(cascade, ctas=None):
        sp = s_pre if ctas is None else s_pre_hi
        append()
        sp.wait_stream(main)
        s_dec.wait_stream(main)
        with torch.cuda.stream(sp):
            prefill(ctas)
        with torch.cuda.stream(s_dec):
            decode_cascade() if cascade else decode()
        main.wait_stream(sp)
        main.wait_stream(s_dec)

    def time_concurrent(cascade, ctas=None, steps=K):
        for _ in range(3):
            concurrent_step(cascade, ctas)
        torch.cuda.synchronize()
        c0, c1 = E(enable_timing=True), E(enable_timing=True)
        c0.record()
        for _ in range(steps):
            concurrent_step(cascade, ctas)
        c1.record()
        torch.cuda.synchronize()
        return c0.elapsed_time(c1) / steps

    t_conc = {cascade: time_concurrent(cascade) for cascade in (False, True)}
    split_sweep = {c: round(time_concurrent(True, c), 4) for c in (72, 80, 88, 96, 104, 120, 136)}
    best_ctas = min(split_sweep, key=split_sweep.get)
    t_split = time_concurrent(True, best_ctas)
    # the same step over an FP8 (e4m3) cache: quantizing append, prefill
    # (pages widened to bf16 in a workspace, then the tensor-core prefill),
    # FP8 decode
    ks8, vs8 = 0.03125, 0.03125
    kc8, vc8 = wl.fp8_pools(w, ks8, vs8)
    pws8 = torch.empty(pagedkv.prefill_fp8_workspace_bytes(
        len(plens), w.prefill_tables.shape[1], hkv, d), dtype=torch.uint8, device=dev)

    def fp8_parts():
        yield lambda: pagedkv.kv_append_fp8(w.k_new, w.v_new, w.slot_mapping, kc8, vc8, ks8, vs8)
        yield lambda: pagedkv.paged_prefill_attention_fp8(
            w.q_prefill, w.q_start, kc8, vc8, w.prefill_tables, w.prefill_lens, True, w.scale,
            ks8, vs8, out=pout, max_q_len=chunk, workspace=pws8)
        yield lambda: pagedkv.paged_decode_attention_fp8(
            w.q_decode, kc8, vc8, w.decode_tables, w.decode_lens, w.scale, ks8, vs8, out=dout,
            max_context_len=max_d, workspace=ws)

    parts8 = list(fp8_parts())
    for _ in range(3):
        for f in parts8:
            f()
    torch.cuda.synchronize()
    marks8 = [tuple(E(enable_timing=True) for _ in range(4)) for _ in range(K)]
    for m in marks8:
        for i, f in enumerate(parts8):
            m[i].record()
            f()
        m[3].record()
    torch.cuda.synchronize()
    ms8 = lambda i, j: sum(m[i].elapsed_time(m[j]) for m in marks8) / K  # noqa: E731
    # the FP8 step with the SMs split: the FP8 prefill persistent on at most
    # `ctas` SMs (high-priority stream), the FP8 decode on the others
    def fp8_concurrent(ctas):
        parts8[0]()
        s_pre_hi.wait_stream(main)
        s_dec.wait_stream(main)
        with torch.cuda.stream(s_pre_hi):
            pagedkv.paged_prefill_attention_fp8(
                w.q_prefill, w.q_start, kc8, vc8, w.prefill_tables, w.prefill_lens, True,
                w.scale, ks8, vs8, out=pout, max_q_len=chunk, workspace=pws8, max_ctas=ctas)
        with torch.cuda.stream(s_dec):
            # beside another kernel the decode takes the uniform split, whose
            # CTAs fill whatever SMs are free (the flat split's persistent
            # grid wants its SMs to itself)
            pagedkv.paged_decode_attention_fp8(
                w.q_decode, kc8, vc8, w.decode_tables, w.decode_lens, w.scale, ks8, vs8,
                out=dout, max_context_len=max_d, workspace=ws,
                partition_blocks=pagedkv.SPLIT_UNIFORM)
        main.wait_stream(s_pre_hi)
        main.wait_stream(s_dec)

    def time_fp8_concurrent(ctas, steps=K):
        for _ in range(3):
            fp8_concurrent(ctas)
        torch.cuda.synchronize()
        c0, c1 = E(enable_timing=True), E(enable_timing=True)
        c0.record()
        for _ in range(steps):
            fp8_concurrent(ctas)
        c1.record()
        torch.cuda.synchronize()
        return c0.elapsed_time(c1) / steps

    # the whole step's attention as one persistent launch (prefill tiles and
    # decode runs from one work list), after the append
    mws = pagedkv.mixed_step_workspace(len(plens), w.prefill_tables.shape[1], len(dlens), hq,
                                       hkv, d, max_d, dev)

    # the decodes' shared 1024-token prefix as one prefix group: attended once
    # on the tensor cores inside the same launch
    gws = pagedkv.mixed_step_workspace(len(plens), w.prefill_tables.shape[1], len(dlens), hq,
                                       hkv, d, max_d, dev, num_groups=1)
    groups = (torch.tensor([0, len(dlens)], dtype=torch.int32, device=dev),
              torch.tensor([w.meta["shared_prefix"] // wl.BLOCK_SIZE], dtype=torch.int32,
                           device=dev), len(dlens), w.meta["shared_prefix"] // wl.BLOCK_SIZE)

    def unified_step(span=0, grouped=False):
        append()
        pagedkv.mixed_step_attention(w.q_prefill, w.q_start, w.prefill_tables, w.prefill_lens,
                                     True, w.q_decode, w.decode_tables, w.decode_lens, kc, vc,
                                     w.scale, chunk, max_d, out_prefill=pout, out_decode=dout,
                                     workspace=gws if grouped else mws,
                                     prefill_span_permille=span,
                                     decode_groups=groups if grouped else None)

    def time_unified(span=0, grouped=False, steps=K):
        for _ in range(3):
            unified_step(span, grouped)
        torch.cuda.synchronize()
        c0, c1 = E(enable_timing=True), E(enable_timing=True)
        c0.record()
        for _ in range(steps):
            unified_step(span, grouped)
        c1.record()
        torch.cuda.synchronize()
        return c0.elapsed_time(c1) / steps

    t_unified = time_unified()
    t_unified_grouped = time_unified(grouped=True)
    span_sweep = ({sp: [round(time_unified(sp, g, max(5, K // 3)), 4) for g in (False, True)]
                   for sp in (500, 700, 800, 900, 950, 1000)}
                  if args.mixed_span_sweep else None)
    del mws, gws
    fp8_sweep = {c: round(time_fp8_concurrent(c), 4) for c in (88, 96, 104, 112, 120)}
    fp8_best = min(fp8_sweep, key=fp8_sweep.get)
    fp8_step = {"ms_per_step": round(ms8(0, 3), 4), "append_ms": round(ms8(0, 1), 4),
                "prefill_ms": round(ms8(1, 2), 4), "decode_ms": round(ms8(2, 3), 4),
                "k_scale": ks8, "v_scale": vs8,
                "prefill_note": "FP8 pages widened in a workspace (K to bf16, V to f16, exact), "
                                "then the tcgen05 prefill with P as one f16 operand and "
                                "k_scale/v_scale folded in",
                "gpu_launches": K * (4 + (1 if ws is not None else 0)),
                "two_streams_sm_split": {
                    "ms_per_step": round(time_fp8_concurrent(fp8_best), 4),
                    "prefill_ctas": fp8_best, "sweep_ms_by_prefill_ctas": fp8_sweep,
                    "note": "FP8 decode on the SMs the persistent FP8 prefill leaves free"}}
    del kc8, vc8, pws8
    flops = prefill_flops(plens, [chunk] * len(plens)) * 4 * hq * d
    row = 2 * hkv * d * 2
    dec_logical = sum(dlens) * row
    prefix_blocks = w.meta["shared_prefix"] // wl.BLOCK_SIZE
    dec_unique = dec_logical - (len(dlens) - 1) * prefix_blocks * wl.BLOCK_SIZE * row
    pre_kv = sum(plens) * row
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except (OSError, ValueError):
        pass
    tflops_peak = float(peaks.get("bf16_tflops", 1900.0))
    hbm, _ = measured_peak()
    t_roof = (dec_unique + pre_kv) / (hbm * 1e9) + flops / (tflops_peak * 1e12)
    cpu = None
    if getattr(args, "mixed_cpu_seconds", 0) > 0:
        # the oracle on a sample of the same step: whole decode sequences
        # (append + decode), and the first, a middle and the last 128-row
        # query tile of prefill chunks; the full step's CPU time is
        # extrapolated from the two rates (KV bytes and FLOPs)
        P = len(plens)
        dview = wl.DecodeWorkload("mixed decodes", w.q_decode, kc, vc, w.k_new[P * chunk:],
                                  w.v_new[P * chunk:], w.slot_mapping[P * chunk:],
                                  w.decode_tables, w.decode_lens, w.scale,
                                  {"lens": dlens})
        dorder = sorted(range(len(dlens)), key=lambda i: (i % 8, i))
        dec_gbps, dinfo = cpu_oracle_sample(dview, args.mixed_cpu_seconds / 2, dorder)
        tiles = [(0, 16), (chunk // 2 - 16, chunk // 2), (chunk - 16, chunk)]
        pre_gflops, pwall, pflops = cpu_prefill_sample(w, range(P), tiles,
                                                       args.mixed_cpu_seconds / 2)
        cpu_ms = (dec_logical / (dec_gbps * 1e9) + flops / (pre_gflops * 1e9)) * 1e3
        cpu = {"value": round(cpu_ms, 1), "unit": "ms per step (extrapolated)",
               "cores": dinfo["cores"], "kind": "oracle",
               "decode_GBps": round(dec_gbps, 4), "prefill_GFLOPs": round(pre_gflops, 3),
               "sample": f"{dinfo['sample']}; prefill: 3 query tiles (16 tokens x 64 heads) "
                         f"of chunks until {args.mixed_cpu_seconds / 2:.0f} s "
                         f"({pflops / 1e9:.1f} GFLOP in {pwall:.1f} s), numpy float64"}
    return {
        "workload": w.name, "steps": K, "ms_per_step": round(t_step, 4),
        "append_ms": round(t_app, 4), "prefill_ms": round(t_pre, 4),
        "decode_ms": round(t_dec, 4),
        "new_tokens": int(w.slot_mapping.shape[0]),
        "prefill": {"kernel": "V pages to f16 + paged_prefill_kernel<128,8,f16 PV> (tcgen05)",
                    "bound": "tensor",
                    "flops_per_launch": flops, "achieved": round(flops / (t_pre / 1e3) / 1e12, 1),
                    "peak": tflops_peak, "unit": "TFLOP/s",
                    "frac": round(flops / (t_pre / 1e3) / 1e12 / tflops_peak, 4),
                    "peak_kind": "measured bf16 burst",
                    "plain_entry_point_ms": round(t_pre_plain, 4),
                    "plain_entry_point_frac": round(flops / (t_pre_plain / 1e3) / 1e12 / tflops_peak,
                                                    4)},
        "decode": {"logical_kv_bytes": dec_logical, "unique_kv_bytes": dec_unique,
                   "logical_GBps": round(dec_logical / (t_dec / 1e3) / 1e9, 1),
                   "unique_GBps": round(dec_unique / (t_dec / 1e3) / 1e9, 1)},
        "decode_shared_prefix": {
            "ms": round(t_casc, 4),
            "unique_GBps": round(dec_unique / (t_casc / 1e3) / 1e9, 1),
            "note": "prefix attended once (tensor cores, beside the private pages) + private "
                    "pages on the library's split (flat for this batch) + LSE merge"},
        "ms_per_step_shared_prefix": round(t_app + t_pre + t_casc, 4),
        "ms_per_step_two_streams": round(t_conc[False], 4),
        "ms_per_step_two_streams_shared_prefix": round(t_conc[True], 4),
        "two_streams_sm_split": {
            "ms_per_step": round(t_split, 4), "prefill_ctas": best_ctas,
            "sweep_ms_by_prefill_ctas": split_sweep,
            "note": "shared-prefix decode on the SMs the persistent prefill leaves free; its "
                    "flat split wants all but 16 SMs to itself, so beside the prefill its "
                    "late CTAs set the time -- the fused launch is the concurrent path"},
        "unified": {
            "ms_per_step": round(t_unified_grouped, 4),
            "frac_of_roofline": round(t_roof * 1e3 / t_unified_grouped, 4),
            "ms_per_step_without_prefix_group": round(t_unified, 4),
            "sweep_ms_by_prefill_span_permille": span_sweep,
            "note": "append, then pkv_mixed_step_attention_ex with the decodes' shared prefix "
                    "as one prefix group: V pages to f16, the prefix check, the decode plan, "
                    "one persistent launch of prefix tiles, prefill tiles and decode runs "
                    "from one work list, the decode merge"},
        "gpu_launches": K * (4 + (1 if ws is not None else 0)),
        "roofline_step_ms": round(t_roof * 1e3, 4),
        "step_frac_of_roofline": round(t_roof * 1e3 / t_step, 4),
        "fp8_cache": fp8_step,
        "cpu_baseline": cpu,
    }


def run_prefill_lengths(dev, pagedkv, E, steps=20):
    """The tensor-core prefill (workspace path: f16 P; plain entry point:
    bf16 hi + lo P) of 64/8-head, d 128 causal chunks over growing cached
    contexts: the mixed step's 8 chunks of 512 tokens, 8 chunks of 512 after
    1K, 16K and 32K cached tokens, and 2 chunks of 4096 from an empty cache.
    A CTA's work (two 128-row query tiles against every key they see) grows
    with the context, so the rows separate the steady tile rate from the
    per-CTA start and end."""
    hq, hkv, d = 64, 8, 128
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except (OSError, ValueError):
        pass
    tflops_peak = float(peaks.get("bf16_tflops", 1900.0))
    cases = (("mixed-step chunks", wl.mixed_prefill_priors(), [512] * 8),
             ("8 x 512 after 1K", [1024] * 8, [512] * 8),
             ("8 x 512 after 16K", [16384] * 8, [512] * 8),
             ("8 x 512 after 32K", [32768] * 8, [512] * 8),
             ("2 x 4096 from empty", [0, 0], [4096, 4096]))
    rows = []
    for name, priors, chunks in cases:
        w = wl.make_chunked_workload(hq, hkv, d, priors, chunks, device=dev, gen_device=dev)
        out = torch.empty(w.q_prefill.shape, dtype=torch.float32, device=dev)
        ws = pagedkv.prefill_workspace(len(priors), w.prefill_tables.shape[1], hkv, d, dev)
        flops = 4 * d * hq * prefill_flops([p + n for p, n in zip(priors, chunks)], chunks)
        row = {"case": name, "gflop": round(flops / 1e9, 1)}
        for path, wsp in (("workspace", ws), ("plain", None)):
            def call():
                pagedkv.paged_prefill_attention(w.q_prefill, w.q_start, w.k_cache, w.v_cache,
                                                w.prefill_tables, w.prefill_lens, True, w.scale,
                                                out=out, max_q_len=max(chunks), workspace=wsp)
            for _ in range(5):
                call()
            torch.cuda.synchronize()
            a, b = E(enable_timing=True), E(enable_timing=True)
            a.record()
            for _ in range(steps):
                call()
            b.record()
            torch.cuda.synchronize()
            ms = a.elapsed_time(b) / steps
            tf = flops / (ms * 1e-3) / 1e12
            row[path] = {"ms": round(ms, 4), "TFLOPs": round(tf, 1),
                         "frac": round(tf / tflops_peak, 3)}
        rows.append(row)
        del w, out, ws
        torch.cuda.empty_cache()
    err = pagedkv.get_device_error(clear=True)
    if err:
        raise RuntimeError(f"device error word {err:#x}: {pagedkv.describe_device_error(err)}")
    return {"peak_tflops": tflops_peak, "peak_kind": "measured bf16 burst" if peaks else
            "fallback", "launches_per_row": steps, "rows": rows}


def run_fused(args, dev, pagedkv, E):
    """Only the fused continuous-batching step: append every new token, then
    pkv_mixed_step_attention_ex with the decodes' shared prefix as one
    prefix group (profiling runs: few launches besides the fused ones)."""
    w = wl.make_mixed_workload(device=dev, gen_device=dev, num_decode=args.mixed_decodes)
    kc, vc = w.k_cache, w.v_cache
    chunk = w.meta["chunk"]
    plens, dlens = w.meta["prefill_lens"], w.meta["decode_lens"]
    hq, d, hkv = w.q_prefill.shape[1], w.q_prefill.shape[2], kc.shape[2]
    max_d = max(dlens)
    pout = torch.empty(w.q_prefill.shape, dtype=torch.float32, device=dev)
    dout = torch.empty(w.q_decode.shape, dtype=torch.float32, device=dev)
    pb = w.meta["shared_prefix"] // wl.BLOCK_SIZE
    groups = (torch.tensor([0, len(dlens)], dtype=torch.int32, device=dev),
              torch.tensor([pb], dtype=torch.int32, device=dev), len(dlens), pb)
    ws = pagedkv.mixed_step_workspace(len(plens), w.prefill_tables.shape[1], len(dlens), hq, hkv,
                                      d, max_d, dev, num_groups=1)

    def step():
        pagedkv.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
        pagedkv.mixed_step_attention(w.q_prefill, w.q_start, w.prefill_tables, w.prefill_lens,
                                     True, w.q_decode, w.decode_tables, w.decode_lens, kc, vc,
                                     w.scale, chunk, max_d, out_prefill=pout, out_decode=dout,
                                     workspace=ws, decode_groups=groups)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    K = args.mixed_steps
    a, b = E(enable_timing=True), E(enable_timing=True)
    a.record()
    for _ in range(K):
        step()
    b.record()
    torch.cuda.synchronize()
    return {"workload": w.name if args.mixed_decodes is None else
            f"{w.name}, shrunk to {len(dlens)} decodes", "steps": K,
            "ms_per_step": round(a.elapsed_time(b) / K, 4)}


def run_fp8(w, dev, pagedkv, E, args, peak):
    """The same 70B-GQA decode step over an FP8 (e4m3) cache: quantizing
    append + FP8 decode.  KV bytes are the e4m3 codes read (half of bf16)."""
    ks, vs = wl.FP8_SCALES[args.workload]
    kc8, vc8 = wl.fp8_pools(w, ks, vs)
    S, hq, hkv, d = w.num_seqs, w.q_heads, w.kv_heads, w.d_head
    max_len = max(w.meta["lens"])
    ws = pagedkv.decode_workspace(S, hq, hkv, d, max_len, dev)
    out = torch.empty(S, hq, d, dtype=torch.float32, device=dev)

    def step():
        pagedkv.kv_append_fp8(w.k_new, w.v_new, w.slot_mapping, kc8, vc8, ks, vs)
        pagedkv.paged_decode_attention_fp8(w.q, kc8, vc8, w.block_tables, w.context_lens,
                                           w.scale, ks, vs, out=out, max_context_len=max_len,
                                           workspace=ws)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    K = args.steps
    marks = [(E(enable_timing=True), E(enable_timing=True)) for _ in range(K)]
    s0, s1 = E(enable_timing=True), E(enable_timing=True)
    s0.record()
    for a, b in marks:
        pagedkv.kv_append_fp8(w.k_new, w.v_new, w.slot_mapping, kc8, vc8, ks, vs)
        a.record()
        pagedkv.paged_decode_attention_fp8(w.q, kc8, vc8, w.block_tables, w.context_lens,
                                           w.scale, ks, vs, out=out, max_context_len=max_len,
                                           workspace=ws)
        b.record()
    s1.record()
    torch.cuda.synchronize()
    t_step = s0.elapsed_time(s1) / K
    t_dec = sum(a.elapsed_time(b) for a, b in marks) / K
    fp8_bytes = int(w.context_lens.sum().item()) * 2 * hkv * d  # one byte per element
    del kc8, vc8
    return {"k_scale": ks, "v_scale": vs, "ms_per_step": round(t_step, 4),
            "decode_ms": round(t_dec, 4), "kv_bytes_per_step": fp8_bytes,
            "KV_GBps": round(fp8_bytes / (t_step / 1e3) / 1e9, 1),
            "decode_GBps": round(fp8_bytes / (t_dec / 1e3) / 1e9, 1),
            "decode_frac_of_hbm": round(fp8_bytes / (t_dec / 1e3) / 1e9 / peak, 4),
            "decode_tokens_per_s": round(S / (t_step / 1e3), 1),
            "gpu_launches": K * (2 + (1 if ws is not None else 0))}


def run_decode_configs(dev, pagedkv, E, peak, names=("mha7b", "long128k"), steps=50,
                       cpu_seconds=0.0):
    """The other full-size decode workloads (7B-MHA, 128K long context): one
    step = append + split-K decode, KV GB/s and fraction of the HBM peak, and
    (cpu_seconds > 0) the CPU oracle on whole sequences of the same workload."""
    res = {}
    for name in names:
        spec = wl.DECODE_SPECS[name]
        w = wl.make_decode_workload(spec, device=dev, gen_device=dev)
        S, hq, hkv, d = w.num_seqs, w.q_heads, w.kv_heads, w.d_head
        max_len = max(w.meta["lens"])
        plan = pagedkv.decode_plan(S, hq, hkv, d, max_len)
        ws = pagedkv.decode_workspace(S, hq, hkv, d, max_len, dev)
        out = torch.empty(S, hq, d, dtype=torch.float32, device=dev)
        marks = [(E(enable_timing=True), E(enable_timing=True)) for _ in range(steps)]

        def append():
            pagedkv.kv_append(w.k_new, w.v_new, w.slot_mapping, w.k_cache, w.v_cache)

        def decode():
            pagedkv.paged_decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables,
                                           w.context_lens, w.scale, out=out,
                                           max_context_len=max_len, workspace=ws)

        for _ in range(5):
            append(), decode()
        torch.cuda.synchronize()
        s0, s1 = E(enable_timing=True), E(enable_timing=True)
        s0.record()
        for a, b in marks:
            append()
            a.record()
            decode()
            b.record()
        s1.record()
        torch.cuda.synchronize()
        t_step = s0.elapsed_time(s1) / steps
        t_dec = sum(a.elapsed_time(b) for a, b in marks) / steps
        kv = w.kv_bytes()
        res[name] = {"workload": spec.name, "kv_bytes": kv, "ms_per_step": round(t_step, 4),
                     "decode_ms": round(t_dec, 4),
                     "KV_GBps": round(kv / (t_step / 1e3) / 1e9, 1),
                     "decode_GBps": round(kv / (t_dec / 1e3) / 1e9, 1),
                     "decode_frac_of_hbm": round(kv / (t_dec / 1e3) / 1e9 / peak, 4),
                     "decode_tokens_per_s": round(S / (t_step / 1e3), 1),
                     "partition_blocks": plan[0], "num_parts": plan[1]}
        if cpu_seconds > 0:
            # spread over the batch: first, middle and last sequences first
            order = sorted(range(S), key=lambda i: (i % max(1, S // 4), i))
            _, info = cpu_oracle_sample(w, cpu_seconds, order)
            res[name]["cpu_baseline"] = info
        del w, ws, out
        torch.cuda.empty_cache()
    return res


def run_append_probe(dev, pagedkv, E, peak, tokens=262144, steps=20):
    """Bulk KV append: `tokens` (default 262,144) of the 70B-GQA row shape (8
    KV heads x 128, 4096 B of K+V per token in bf16) scattered to random slots
    of a pool 1.25x their size.  Bytes = rows read + rows written."""
    hkv, d = 8, 128
    g = torch.Generator(device=dev).manual_seed(7001)
    k = torch.randn(tokens, hkv, d, generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn(tokens, hkv, d, generator=g, device=dev).to(torch.bfloat16)
    nb = (tokens * 5 // 4 + wl.BLOCK_SIZE - 1) // wl.BLOCK_SIZE
    slots = torch.randperm(nb * wl.BLOCK_SIZE, generator=torch.Generator().manual_seed(7002))
    slots = slots[:tokens].to(dev)
    kc = torch.empty(nb, wl.BLOCK_SIZE, hkv, d, dtype=torch.bfloat16, device=dev)
    vc = torch.empty_like(kc)
    kc8 = torch.empty(kc.shape, dtype=torch.uint8, device=dev)
    vc8 = torch.empty_like(kc8)
    res = {"tokens": tokens}
    for name, fn, row_bytes in (
            ("bf16", lambda: pagedkv.kv_append(k, v, slots, kc, vc), 2 * hkv * d * 2),
            ("fp8", lambda: pagedkv.kv_append_fp8(k, v, slots, kc8, vc8, 0.03125, 0.03125),
             2 * hkv * d * 2 + 2 * hkv * d)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = E(enable_timing=True), E(enable_timing=True)
        a.record()
        for _ in range(steps):
            fn()
        b.record()
        torch.cuda.synchronize()
        t = a.elapsed_time(b) / steps
        moved = tokens * (row_bytes if name == "fp8" else 2 * row_bytes)
        res[name] = {"ms": round(t, 4), "bytes_moved": moved,
                     "GBps": round(moved / (t / 1e3) / 1e9, 1),
                     "frac_of_hbm": round(moved / (t / 1e3) / 1e9 / peak, 4)}
    del k, v, kc, vc, kc8, vc8
    torch.cuda.empty_cache()
    return res


def run_small_batch(dev, pagedkv, E, batches=(1, 2, 4, 8, 16, 32, 64), steps=200,
                    short_len=512):
    """Small-batch decode steps of the 70B-GQA layer shape: per-step time of
    eager calls vs replay of a CUDA graph captured for the batch's bucket
    (the decode step: append + decode, the library's split: uniform, or flat
    for 25-128 sequences).  Batches of 1-4 sequences have short contexts
    (`short_len` tokens each), where launch latency dominates; 8 to 64 draw
    their contexts from the 70B-GQA recipe."""
    from paged_kv_cache_52_gb300.graphs import DecodeGraphRunner
    res = {}
    for bsz in batches:
        lens = [short_len] * bsz if bsz <= 4 else None
        w = wl.make_decode_workload(wl.GQA_70B, device=dev, gen_device=dev,
                                    num_seqs_override=bsz, lens_override=lens)
        max_len = max(w.meta["lens"])
        ws = pagedkv.decode_workspace(bsz, w.q_heads, w.kv_heads, w.d_head, max_len, dev)
        out = torch.empty(w.q.shape, dtype=torch.float32, device=dev)

        def eager():
            pagedkv.paged_decode_step(w.q, w.k_new, w.v_new, w.slot_mapping, w.k_cache,
                                      w.v_cache, w.block_tables, w.context_lens, w.scale, out=out,
                                      max_context_len=max_len, workspace=ws)

        runner = DecodeGraphRunner(w.k_cache, w.v_cache, w.q_heads, w.block_tables.shape[1],
                                   max_len, w.scale, buckets=(bsz,))
        b = runner.capture(bsz)
        b.q.copy_(w.q), b.k_new.copy_(w.k_new), b.v_new.copy_(w.v_new)
        b.slots.copy_(w.slot_mapping), b.tables.copy_(w.block_tables), b.lens.copy_(w.context_lens)
        times = {}
        for name, fn in (("eager", eager), ("graph", b.graph.replay)):
            for _ in range(10):
                fn()
            torch.cuda.synchronize()
            s0, s1 = E(enable_timing=True), E(enable_timing=True)
            s0.record()
            for _ in range(steps):
                fn()
            s1.record()
            torch.cuda.synchronize()
            times[name] = s0.elapsed_time(s1) / steps * 1e3
        flat = pagedkv.decode_plan_uses_flat(bsz, w.q_heads, w.kv_heads, w.d_head, max_len, 0)
        res[str(bsz)] = {"eager_us": round(times["eager"], 2), "graph_us": round(times["graph"], 2),
                         "context_lens": "512 each" if lens else "U[1024, 8192]",
                         "kv_bytes": w.kv_bytes(), "split": "flat" if flat else "uniform",
                         "graph_GBps": round(w.kv_bytes() / (times["graph"] / 1e6) / 1e9, 1)}
        del w, runner, b
    return res



def e2e_pipelined(host, w, K, step, out, ws, max_len, args, dev, pagedkv, barrier):
    """K steps through the public API with host buffers: step i's inputs go up
    on a copy stream while step i-1 computes, and its output comes back while
    step i+1 computes.  Two sets of device inputs and outputs, ordered by
    events; every step still moves all of its inputs and its output."""
    comp = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(dev)
    E = torch.cuda.Event
    devb = [{n: torch.empty_like(getattr(w, n)) for n in host} for _ in range(2)]
    outs = [torch.empty_like(out) for _ in range(2)]
    outs_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    uploaded = [E() for _ in range(2)]
    computed = [E() for _ in range(2)]
    read_back = [E() for _ in range(2)]
    kc, vc = w.k_cache, w.v_cache

    def upload(i):
        b = i % 2
        with torch.cuda.stream(copy):
            copy.wait_event(computed[b])     # step i-2 is done with this set
            for n, t in host.items():
                devb[b][n].copy_(t, non_blocking=True)
            uploaded[b].record(copy)

    def run(steps):
        for b in range(2):
            computed[b].record(comp)
            read_back[b].record(comp)
        upload(0)
        for i in range(steps):
            b = i % 2
            if i + 1 < steps:
                upload(i + 1)
            comp.wait_event(uploaded[b])
            comp.wait_event(read_back[b])    # step i-2's output has left this buffer
            d = devb[b]
            step(d["k_new"], d["v_new"], d["slot_mapping"], d["q"], d["block_tables"],
                 d["context_lens"], outs[b])
            computed[b].record(comp)
            with torch.cuda.stream(copy):
                copy.wait_event(computed[b])
                outs_h[b].copy_(outs[b], non_blocking=True)
                read_back[b].record(copy)
        comp.wait_event(read_back[(steps - 1) % 2])
        if steps > 1:
            comp.wait_event(read_back[(steps - 2) % 2])

    run(3)
    torch.cuda.synchronize()
    barrier()
    s, e = E(enable_timing=True), E(enable_timing=True)
    s.record(comp)
    copy.wait_event(s)
    run(K)
    e.record(comp)
    torch.cuda.synchronize()
    torch.testing.assert_close(outs_h[(K - 1) % 2], out.cpu(), rtol=0, atol=0)
    return max_over_ranks(s.elapsed_time(e), dev)

def run_verify(dev, pagedkv, E, peak, num_seqs=256):
    """Speculative verification at the 70B-GQA decode shape: 256 sequences,
    K drafted tokens each (already appended), contexts U[1024, 8192].  The
    multi-query decode kernel against the same attention through the chunked
    prefill kernel (K-token causal chunks).  KV bytes are those of the decode."""
    g = torch.Generator().manual_seed(3005)
    lens = torch.randint(1024, 8193, (num_seqs,), generator=g).tolist()
    res = {"num_seqs": num_seqs}
    for K in (2, 4):
        w = wl.make_chunked_workload(64, 8, 128, [L - K for L in lens], [K] * num_seqs,
                                     config_id=9, device=dev, gen_device=dev)
        S, hq, d = num_seqs, 64, 128
        q = w.q_prefill.view(S, K, hq, d)
        max_len = max(lens)
        ws = pagedkv.verify_workspace(S, K, hq, 8, d, max_len, dev)
        out = torch.empty(S, K, hq, d, dtype=torch.float32, device=dev)
        pout = torch.empty(w.q_prefill.shape, dtype=torch.float32, device=dev)
        calls = {
            "verify_kernel": lambda: pagedkv.paged_verify_attention(
                q, w.k_cache, w.v_cache, w.prefill_tables, w.prefill_lens, w.scale, out=out,
                max_context_len=max_len, workspace=ws),
            "prefill_kernel": lambda: pagedkv.paged_prefill_attention(
                w.q_prefill, w.q_start, w.k_cache, w.v_cache, w.prefill_tables, w.prefill_lens,
                True, w.scale, out=pout, max_q_len=K),
        }
        kv = sum(lens) * 2 * 8 * d * 2
        row = {"kv_bytes": kv}
        for name, f in calls.items():
            for _ in range(3):
                f()
            torch.cuda.synchronize()
            a, b = E(enable_timing=True), E(enable_timing=True)
            a.record()
            for _ in range(20):
                f()
            b.record()
            torch.cuda.synchronize()
            t = a.elapsed_time(b) / 20
            row[name] = {"ms": round(t, 4), "GBps": round(kv / (t / 1e3) / 1e9, 1),
                         "frac_of_hbm": round(kv / (t / 1e3) / 1e9 / peak, 4)}
        row["tokens_verified_per_s"] = round(S * K / (row["verify_kernel"]["ms"] / 1e3), 1)
        res[f"K{K}"] = row
        del w, q, out, pout, ws
        torch.cuda.empty_cache()
    return res


def run_ours(args):
    rank, world, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from paged_kv_cache_52_gb300 import pagedkv

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    if args.only_mixed:
        print(json.dumps({"mixed_step": run_mixed(args, dev, pagedkv, torch.cuda.Event)}))
        return
    if args.only_fused:
        print(json.dumps({"fused_mixed_step": run_fused(args, dev, pagedkv, torch.cuda.Event)}))
        return
    if args.only_prefill_lengths:
        print(json.dumps({"prefill_lengths": run_prefill_lengths(dev, pagedkv, torch.cuda.Event)}))
        return
    if args.only_append:
        peak, _ = measured_peak()
        print(json.dumps({"append_probe": run_append_probe(dev, pagedkv, torch.cuda.Event, peak,
                                                           args.append_tokens,
                                                           args.append_steps)}))
        return
    if args.only_verify:
        peak, _ = measured_peak()
        print(json.dumps({"speculative_verify": run_verify(dev, pagedkv, torch.cuda.Event, peak,
                                                           args.verify_seqs)}))
        return
    spec = wl.DECODE_SPECS[args.workload]
    w = wl.make_decode_workload(spec, device=dev, gen_device=dev,
                                num_seqs_override=args.num_seqs or None)
    S, hq, hkv, d = w.num_seqs, w.q_heads, w.kv_heads, w.d_head
    max_len = max(w.meta["lens"])
    plan = pagedkv.decode_plan(S, hq, hkv, d, max_len, args.partition_blocks)
    ws = pagedkv.decode_workspace(S, hq, hkv, d, max_len, dev, args.partition_blocks)
    out = torch.empty(S, hq, d, dtype=torch.float32, device=dev)
    kc, vc = w.k_cache, w.v_cache
    kv_bytes = w.kv_bytes()

    def append(k_new, v_new, slots):
        pagedkv.kv_append(k_new, v_new, slots, kc, vc)

    def decode(q, tables, lens):
        pagedkv.paged_decode_attention(q, kc, vc, tables, lens, w.scale, out=out,
                                       max_context_len=max_len, workspace=ws,
                                       partition_blocks=args.partition_blocks)

    def step(k_new, v_new, slots, q, tables, lens, dst=None):
        """One decode step through the public API: the new token of every
        sequence appended, then attended (pkv_paged_decode_step, which hides
        the append under the attention; --separate-step: the two calls)."""
        dst = out if dst is None else dst
        if args.separate_step or args.partition_blocks:
            append(k_new, v_new, slots)
            pagedkv.paged_decode_attention(q, kc, vc, tables, lens, w.scale, out=dst,
                                           max_context_len=max_len, workspace=ws,
                                           partition_blocks=args.partition_blocks)
        else:
            pagedkv.paged_decode_step(q, k_new, v_new, slots, kc, vc, tables, lens, w.scale,
                                      out=dst, max_context_len=max_len, workspace=ws)

    inputs = (w.k_new, w.v_new, w.slot_mapping, w.q, w.block_tables, w.context_lens)
    for _ in range(max(3, args.warmup)):
        step(*inputs)
    torch.cuda.synchronize()
    err = pagedkv.get_device_error(clear=True)
    if err:
        raise RuntimeError(f"device error word {err:#x}: {pagedkv.describe_device_error(err)}")

    K = args.steps
    E = torch.cuda.Event
    start, end = E(enable_timing=True), E(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        # keep the GPU under the same load while nvidia-smi starts sampling,
        # so the samples bracket the timed region
        t_load = time.perf_counter()
        while time.perf_counter() - t_load < 0.6:
            for _ in range(50):
                step(*inputs)
            torch.cuda.synchronize()
        start.record()
        for _ in range(K):
            step(*inputs)
        end.record()
        torch.cuda.synchronize()
    barrier()
    total_ms = max_over_ranks(start.elapsed_time(end), dev)
    ms_per_step = total_ms / K
    value = whole_job_gbps(kv_bytes, K, world, total_ms)
    # the step's parts, each call timed alone: the append, and the decode
    # call whose bytes the roofline counts
    marks = [(E(enable_timing=True), E(enable_timing=True), E(enable_timing=True))
             for _ in range(K)]
    s0, s1 = E(enable_timing=True), E(enable_timing=True)
    s0.record()
    for a, b, c in marks:
        a.record()
        append(w.k_new, w.v_new, w.slot_mapping)
        b.record()
        decode(w.q, w.block_tables, w.context_lens)
        c.record()
    s1.record()
    torch.cuda.synchronize()
    decode_ms = sum(b.elapsed_time(c) for _, b, c in marks) / K
    append_ms = sum(a.elapsed_time(b) for a, b, _ in marks) / K
    separate_ms = s0.elapsed_time(s1) / K

    # End to end through the public API: this step's inputs from pinned host
    # memory, the step, and the output read back, every step.
    host = {n: getattr(w, n).cpu().pin_memory() for n in
            ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens")}
    devb = {n: torch.empty_like(getattr(w, n)) for n in host}
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * out_h.element_size()

    def e2e_step():
        for n, t in host.items():
            devb[n].copy_(t, non_blocking=True)
        step(devb["k_new"], devb["v_new"], devb["slot_mapping"], devb["q"],
             devb["block_tables"], devb["context_lens"])
        out_h.copy_(out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    s2, e2 = E(enable_timing=True), E(enable_timing=True)
    s2.record()
    for _ in range(K):
        e2e_step()
    e2.record()
    torch.cuda.synchronize()
    e2e_serial_ms = max_over_ranks(s2.elapsed_time(e2), dev)
    e2e_ms = e2e_pipelined(host, w, K, step, out, ws, max_len, args, dev, pagedkv, barrier)
    e2e_value = whole_job_gbps(kv_bytes, K, world, e2e_ms)

    peak, peak_kind = measured_peak()
    achieved = kv_bytes / (decode_ms / 1e3) / 1e9
    traffic, _ = read_traffic(args.workload)
    launches_per_step = 2 + (1 if plan[1] > 1 else 0)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": max(3, args.warmup), "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded randn bf16 K/V/q, random block tables (no dataset)",
        "config": workload_config(w, spec, plan),
        "decode_tokens_per_s": round(world * S * K / (total_ms / 1e3), 1),
        # one token per sequence through 80 such attention layers; excludes
        # the weights' matmuls and every other part of a real model step
        "decode_tokens_per_s_80_layers_attention_only": round(
            world * S * K / (80 * total_ms / 1e3), 1),
        "decode_ms": round(decode_ms, 4), "append_ms": round(append_ms, 4),
        "ms_per_step_separate_calls": round(separate_ms, 4),
        "frac_of_nominal_8tbs": round(value / world / NOMINAL_HBM_GBS, 4),
        "roofline": {"kernel": "paged_decode (split-K kernel + LSE merge, one call)",
                     "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": f"{peak_kind} (copy GB/s)", "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes_per_launch": kv_bytes},
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms / K, 4),
                "mode": "pipelined: each step's inputs uploaded from pinned host memory and "
                        "its output read back on a copy stream, double-buffered, so the "
                        "copies of steps i+1 and i-1 overlap the compute of step i",
                "serial": {"value": round(whole_job_gbps(kv_bytes, K, world, e2e_serial_ms), 1),
                           "ms_per_step": round(e2e_serial_ms / K, 4),
                           "mode": "copy in, step, copy out on one stream"}},
        "gpu_launches": launches_per_step * K,
        "clocks": clk.summary(),
    }
    line["fp8_cache"] = run_fp8(w, dev, pagedkv, E, args, peak)
    cpu_here = rank == 0 and world == 1 and not args.no_cpu_baseline
    args.mixed_cpu_seconds = args.config_cpu_seconds if cpu_here else 0.0
    if not args.no_mixed:
        line["other_decode_workloads"] = run_decode_configs(
            dev, pagedkv, E, peak, cpu_seconds=args.mixed_cpu_seconds)
        line["append_probe"] = run_append_probe(dev, pagedkv, E, peak)
    if not args.no_mixed:
        del host, devb
        line["mixed_step"] = run_mixed(args, dev, pagedkv, E)
        line["small_batch_decode"] = run_small_batch(dev, pagedkv, E)
        line["speculative_verify"] = run_verify(dev, pagedkv, E, peak)
    if cpu_here:
        _, info = cpu_oracle_sample(w, args.cpu_seconds)
        line["cpu_baseline"] = info
    line["per_config"] = per_config_summary(line, peak)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def per_config_summary(line, peak):
    """A compact per-config digest, printed last so that a reader keeping only
    the end of the JSON line still sees every workload's headline numbers and
    its CPU oracle baseline."""
    def r(x, n=1):
        return None if x is None else round(x, n)

    def cpu_of(d):
        c = d.get("cpu_baseline") if d else None
        return None if not c else r(c.get("value"), 4)

    out = {"peak_GBps": peak,
           "gqa70b": {"step_GBps": line.get("value"), "decode_frac": line["roofline"]["frac"],
                      "tok_s": line.get("decode_tokens_per_s"),
                      "tok_s_80_layers_attn_only":
                          line.get("decode_tokens_per_s_80_layers_attention_only"),
                      "cpu_GBps": cpu_of(line)}}
    for name, d in (line.get("other_decode_workloads") or {}).items():
        out[name] = {"decode_GBps": d.get("decode_GBps"), "decode_frac": d.get("decode_frac_of_hbm"),
                     "tok_s": d.get("decode_tokens_per_s"), "cpu_GBps": cpu_of(d)}
    fp8 = line.get("fp8_cache")
    if fp8:
        out["gqa70b_fp8"] = {"decode_GBps": fp8.get("decode_GBps"),
                             "decode_frac": fp8.get("decode_frac_of_hbm")}
    m = line.get("mixed_step")
    if m:
        out["mixed"] = {"ms": m["ms_per_step"], "roofline_ms": m["roofline_step_ms"],
                        "prefill_frac": m["prefill"]["frac"],
                        "plain_prefill_frac": m["prefill"]["plain_entry_point_frac"],
                        "decode_unique_GBps": m["decode"]["unique_GBps"],
                        "sm_split_ms": m["two_streams_sm_split"]["ms_per_step"],
                        "cpu_ms": cpu_of(m)}
        if "unified" in m:
            out["mixed"]["fused_ms"] = m["unified"]["ms_per_step"]
    sb = line.get("small_batch_decode")
    if sb:
        out["small_batch_us"] = {k: [v["eager_us"], v["graph_us"]] for k, v in sb.items()}
    return out


def run_reference(args):
    """The oracle on the host cores, on the same metric: each step is the
    append + decode of a bounded sample of the workload's sequences."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle  # the reference arm of this benchmark is the CPU oracle

    spec = wl.DECODE_SPECS[args.workload]
    if spec.lens is not None:
        all_lens = list(spec.lens)
    else:
        lo, hi = spec.len_range
        g = torch.Generator().manual_seed(1000 * spec.config_id + 5)
        all_lens = torch.randint(lo, hi + 1, (spec.num_seqs,), generator=g).tolist()
    per_step = 4 if max(all_lens) <= 16384 else 1
    sample = all_lens[:per_step]
    w = wl.make_decode_workload(spec, lens_override=sample)
    kc0, vc0 = wl.bf16_bits(w.k_cache), wl.bf16_bits(w.v_cache)
    kn, vn = wl.bf16_bits(w.k_new), wl.bf16_bits(w.v_new)
    q = wl.bf16_bits(w.q)
    slots = w.slot_mapping.numpy()
    tables = w.block_tables.numpy()
    kv_bytes = w.kv_bytes()

    def step():
        kc, vc = oracle.kv_append(kn, vn, slots, kc0, vc0)
        oracle.paged_decode_attention(q, kc, vc, tables, sample, w.scale)

    for _ in range(args.warmup):
        step()
    c0, t0 = time.process_time(), time.perf_counter()
    for _ in range(args.steps):
        step()
    wall = time.perf_counter() - t0
    cpu = time.process_time() - c0
    value = kv_bytes * args.steps / wall / 1e9
    cores = max(1, round(cpu / wall))
    desc = (f"oracle append+decode of {per_step} of {spec.num_seqs} sequences per step "
            f"(context lens {sample}), numpy float64")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(wall / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: seeded randn bf16 K/V/q, random block tables (no dataset)",
        "config": {"workload": spec.name, "sample_seqs": per_step, "sample_context_lens": sample,
                   "kv_bytes_per_step": kv_bytes},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores,
                         "kind": "oracle", "host_cpus": len(os.sched_getaffinity(0)),
                         "sample": desc},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
