"""Shared helpers of the parity tests (GPU path vs the CPU oracle).

Tolerance for attention outputs (float32 out of bf16 inputs with float32
softmax accumulation): every element within 2e-3 absolute, and every output
row (one token, one query head) within 1e-2 relative in the 2-norm,
``||gpu - ref|| / max(||ref||, 1e-6)``.  The row-wise relative form is used
because an element-wise relative error is undefined where the exact output
crosses zero.
"""

import numpy as np
import torch

import oracle
from paged_kv_cache_52_gb300 import workloads as wl

ATOL = 2e-3
ROW_RTOL = 1e-2


def attention_errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if got.size == 0:
        return 0.0, 0.0
    max_abs = float(np.abs(got - ref).max())
    d = got.reshape(-1, got.shape[-1]) - ref.reshape(-1, ref.shape[-1])
    rn = np.linalg.norm(ref.reshape(-1, ref.shape[-1]), axis=1)
    row_rel = float((np.linalg.norm(d, axis=1) / np.maximum(rn, 1e-6)).max())
    return max_abs, row_rel


def assert_attention_close(got, ref, what=""):
    got = np.asarray(got)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    max_abs, row_rel = attention_errors(got, ref)
    assert max_abs <= ATOL and row_rel <= ROW_RTOL, \
        f"{what}: max|diff| {max_abs:.3e} (<= {ATOL}), row rel {row_rel:.3e} (<= {ROW_RTOL})"
    return max_abs, row_rel


def compact_pool(k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                 lens, seqs):
    """Copy only the physical blocks the chosen sequences use to the host and
    renumber their tables (pages may sit anywhere, so the oracle's result does
    not depend on which ids they get).  Returns (k_bits, v_bits, tables, remap)."""
    tables = block_tables.cpu().numpy()
    used = []
    for s in seqs:
        nb = wl.blocks_for(int(lens[s]))
        used.extend(int(b) for b in tables[s, :nb])
    uniq = sorted(set(used))
    remap = {b: i for i, b in enumerate(uniq)}
    idx = torch.tensor(uniq if uniq else [0], dtype=torch.int64, device=k_cache.device)
    kc = wl.bf16_bits(k_cache.index_select(0, idx))
    vc = wl.bf16_bits(v_cache.index_select(0, idx))
    new_tables = np.full((len(seqs), max(1, tables.shape[1])), -1, dtype=np.int64)
    for r, s in enumerate(seqs):
        nb = wl.blocks_for(int(lens[s]))
        new_tables[r, :nb] = [remap[int(b)] for b in tables[s, :nb]]
    return kc, vc, new_tables, remap


def remap_slots(slots, remap, block_size=wl.BLOCK_SIZE):
    out = []
    for s in slots:
        s = int(s)
        out.append(-1 if s < 0 else remap[s // block_size] * block_size + s % block_size)
    return np.array(out, dtype=np.int64)


class DecodeStepOracle:
    """Oracle for one decode step (append, then decode) of the chosen
    sequences, built from a host snapshot taken BEFORE the GPU step runs."""

    def __init__(self, w, seqs):
        self.seqs = list(seqs)
        lens = [int(x) for x in w.context_lens.cpu().tolist()]
        self.lens = [lens[s] for s in self.seqs]
        self.kc, self.vc, self.tables, remap = compact_pool(w.k_cache, w.v_cache, w.block_tables,
                                                            lens, self.seqs)
        sl = w.slot_mapping.cpu().numpy()[self.seqs]
        self.slots = remap_slots(sl, remap)
        idx = torch.tensor(self.seqs, dtype=torch.int64, device=w.q.device)
        self.k_new = wl.bf16_bits(w.k_new.index_select(0, idx))
        self.v_new = wl.bf16_bits(w.v_new.index_select(0, idx))
        self.q = wl.bf16_bits(w.q.index_select(0, idx))
        self.scale = w.scale

    def output(self):
        kc, vc = oracle.kv_append(self.k_new, self.v_new, self.slots, self.kc, self.vc)
        return oracle.paged_decode_attention(self.q, kc, vc, self.tables, self.lens, self.scale)


class PrefillStepOracle:
    """Oracle for a chunked-prefill step (append the chunks, then attend) of
    the chosen sequences, from a host snapshot taken BEFORE the GPU step."""

    def __init__(self, w, seqs, causal=True):
        self.seqs = list(seqs)
        self.causal = causal
        lens = [int(x) for x in w.prefill_lens.cpu().tolist()]
        self.lens = [lens[s] for s in self.seqs]
        self.kc, self.vc, self.tables, remap = compact_pool(w.k_cache, w.v_cache,
                                                            w.prefill_tables, lens, self.seqs)
        qs = w.q_start.cpu().numpy()
        rows = np.concatenate([np.arange(qs[s], qs[s + 1]) for s in self.seqs]).astype(np.int64)
        self.rows = rows
        self.q_start = np.concatenate([[0], np.cumsum([qs[s + 1] - qs[s] for s in self.seqs])])
        slots = w.slot_mapping.cpu().numpy()[rows]
        self.slots = remap_slots(slots, remap)
        idx = torch.tensor(rows, dtype=torch.int64, device=w.q_prefill.device)
        self.k_new = wl.bf16_bits(w.k_new.index_select(0, idx))
        self.v_new = wl.bf16_bits(w.v_new.index_select(0, idx))
        self.q = wl.bf16_bits(w.q_prefill.index_select(0, idx))
        self.scale = w.scale

    def cache(self):
        return oracle.kv_append(self.k_new, self.v_new, self.slots, self.kc, self.vc)

    def output(self):
        kc, vc = self.cache()
        return oracle.paged_prefill_attention(self.q, self.q_start, kc, vc, self.tables, self.lens,
                                              self.causal, self.scale)

    def token_range_output(self, si, a, b):
        """Oracle rows of queries [a, b) of local sequence si's chunk.  Those
        queries are the last b - a positions of the first context_len - n + b
        keys, so they are a causal chunk of that shorter context."""
        kc, vc = self._cache_once()
        n = int(self.q_start[si + 1] - self.q_start[si])
        ctx = self.lens[si] - n + b if self.causal else self.lens[si]
        kk = oracle.gather_sequence_kv(kc, self.tables[si], ctx)
        vv = oracle.gather_sequence_kv(vc, self.tables[si], ctx)
        q0 = int(self.q_start[si])
        return oracle.attention(self.q[q0 + a:q0 + b], kk, vv, self.scale, causal=self.causal)

    def _cache_once(self):
        if not hasattr(self, "_cached"):
            self._cached = self.cache()
        return self._cached

    def rows_output(self, picks):
        """Oracle rows for (local sequence index, query index in its chunk)
        pairs: query i of a causal chunk of n equals a decode over the first
        context_len - n + i + 1 tokens."""
        kc, vc = self.cache()
        out = []
        for si, i in picks:
            n = int(self.q_start[si + 1] - self.q_start[si])
            ctx = self.lens[si] - n + i + 1 if self.causal else self.lens[si]
            qrow = self.q[int(self.q_start[si]) + i][None]
            out.append(oracle.paged_decode_attention(qrow, kc, vc, self.tables[si:si + 1], [ctx],
                                                     self.scale)[0])
        return np.stack(out)
