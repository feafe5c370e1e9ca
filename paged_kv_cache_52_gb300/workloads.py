"""Seeded synthetic inputs for paged-KV attention.

This module only draws random numbers and lays out block tables; it holds none
of the attention arithmetic.  Both the CUDA path (tests, ``bench.py``) and the
CPU oracle's tests take their inputs from here.

Recipe (the same for every workload):

* values are drawn as float32 ``randn`` and rounded once to bf16;
* seeds are ``1000 * config_id + k`` with k = 0 queries, 1 K pool, 2 V pool,
  3 new K rows, 4 new V rows, 5 context lengths, 6 block permutation,
  7 outlier rows;
* the physical pool has ``ceil(1.25 * blocks_needed)`` blocks (or a fixed
  count); a random permutation of the pool ids is consumed in order to fill
  the block tables, so pages sit anywhere; unused blocks keep their random
  contents, which serve as a canary for the append;
* "massive activation" outliers: a seeded choice of ``round(frac * rows)``
  K rows (one row = one token of one KV head) of the pool is multiplied by
  the outlier scale in float32 before the single rounding to bf16;
* every decode sequence appends exactly one token, at position
  ``context_len - 1``; context lengths include it.

Large pools are drawn on the device given (``gen_device``) with torch's
generator for that device, in chunks; small ones on the CPU.  Lengths, block
permutations and outlier rows always come from CPU generators.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional, Sequence

import torch

BLOCK_SIZE = 16


def _cpu_gen(seed: int) -> torch.Generator:
    return torch.Generator(device="cpu").manual_seed(int(seed))


def _dev_gen(seed: int, device) -> torch.Generator:
    return torch.Generator(device=torch.device(device)).manual_seed(int(seed))


def _randn_bf16(shape, seed: int, device, gen_device=None, row_scale=None,
                chunk_elems: int = 1 << 28) -> torch.Tensor:
    """float32 randn rounded once to bf16, drawn on ``gen_device`` (default:
    ``device``).  ``row_scale`` = (flat_row_index, factor, row_len) scales the
    selected rows of the float32 draw before rounding."""
    gen_device = torch.device(gen_device if gen_device is not None else device)
    g = _dev_gen(seed, gen_device)
    numel = math.prod(shape)
    out = torch.empty(numel, dtype=torch.bfloat16, device=gen_device)
    rows_sel = None
    row_len = 1
    if row_scale is not None:
        rows_sel, factor, row_len = row_scale
        rows_sel = torch.sort(rows_sel.to(torch.int64).cpu()).values
    # chunk borders fall on row borders, so a scaled row is never split
    chunk = max(row_len, (chunk_elems // row_len) * row_len)
    start = 0
    while start < numel:
        stop = min(numel, start + chunk)
        x = torch.randn(stop - start, generator=g, dtype=torch.float32, device=gen_device)
        if rows_sel is not None:
            r0, r1 = start // row_len, stop // row_len
            lo = int(torch.searchsorted(rows_sel, r0))
            hi = int(torch.searchsorted(rows_sel, r1))
            if hi > lo:
                sel = (rows_sel[lo:hi] - r0).to(gen_device)
                xv = x.view(-1, row_len)
                xv[sel] = xv[sel] * float(factor)
        out[start:stop] = x.to(torch.bfloat16)
        start = stop
    out = out.view(*shape)
    return out.to(device) if out.device != torch.device(device) else out


def blocks_for(length: int, block_size: int = BLOCK_SIZE) -> int:
    return -(-int(length) // block_size)


def build_block_tables(lens: Sequence[int], perm: torch.Tensor, block_size: int = BLOCK_SIZE,
                       shared_prefix_blocks: int = 0, max_blocks: Optional[int] = None):
    """Fill block tables from the permutation, in sequence order.

    The first ``shared_prefix_blocks`` ids of the permutation are the common
    prefix of every table; each sequence then takes its private blocks in
    turn.  Unused table entries are -1.  Returns (tables int32 [S, max_blocks],
    number of permutation entries consumed)."""
    need = [blocks_for(L, block_size) for L in lens]
    mb = max_blocks if max_blocks is not None else max([1] + need)
    tables = torch.full((len(lens), mb), -1, dtype=torch.int32)
    cursor = shared_prefix_blocks
    shared = perm[:shared_prefix_blocks].to(torch.int32)
    for s, nb in enumerate(need):
        nshared = min(shared_prefix_blocks, nb)
        tables[s, :nshared] = shared[:nshared]
        priv = nb - nshared
        tables[s, nshared:nb] = perm[cursor:cursor + priv].to(torch.int32)
        cursor += priv
    return tables, cursor


def append_slots(tables: torch.Tensor, positions: Sequence[Sequence[int]],
                 block_size: int = BLOCK_SIZE) -> torch.Tensor:
    """slot of logical position j of sequence s: table[s][j // bs] * bs + j % bs."""
    slots = []
    for s, pos in enumerate(positions):
        for j in pos:
            slots.append(int(tables[s, j // block_size]) * block_size + j % block_size)
    return torch.tensor(slots, dtype=torch.int64)


@dataclass
class DecodeWorkload:
    """One decode step: append one token per sequence, then attend."""
    name: str
    q: torch.Tensor               # [S, Hq, d] bf16
    k_cache: torch.Tensor         # [NB, bs, Hkv, d] bf16 (before the append)
    v_cache: torch.Tensor
    k_new: torch.Tensor           # [S, Hkv, d] bf16 (the token at position L-1)
    v_new: torch.Tensor
    slot_mapping: torch.Tensor    # [S] int64
    block_tables: torch.Tensor    # [S, max_blocks] int32
    context_lens: torch.Tensor    # [S] int32 (include the appended token)
    scale: float
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self):
        return self.q.shape[0]

    @property
    def q_heads(self):
        return self.q.shape[1]

    @property
    def kv_heads(self):
        return self.k_cache.shape[2]

    @property
    def d_head(self):
        return self.k_cache.shape[3]

    def kv_bytes(self) -> int:
        """Logical K+V bytes the decode reads (every context token, bf16)."""
        return int(self.context_lens.sum().item()) * 2 * self.kv_heads * self.d_head * 2


@dataclass(frozen=True)
class DecodeSpec:
    name: str
    config_id: int
    num_seqs: int
    q_heads: int
    kv_heads: int
    d_head: int
    lens: Optional[tuple] = None          # fixed context lengths
    len_range: Optional[tuple] = None     # inclusive uniform range
    num_blocks: Optional[int] = None      # fixed pool size
    outlier_frac: float = 0.0
    outlier_scale: float = 100.0
    scale: Optional[float] = None         # default 1/sqrt(d)


TINY = DecodeSpec("tiny paged decode (4 seqs, 8/2 heads, d64)", 1, 4, 8, 2, 64,
                  lens=(17, 64, 100, 250), num_blocks=64)
MHA_7B = DecodeSpec("7B-MHA decode layer (64 seqs, 32/32 heads, d128, L~U[512,4096])", 2,
                    64, 32, 32, 128, len_range=(512, 4096))
GQA_70B = DecodeSpec("70B-GQA decode layer (256 seqs, 64/8 heads, d128, L~U[1024,8192], "
                     "0.1% K rows x100)", 3, 256, 64, 8, 128, len_range=(1024, 8192),
                     outlier_frac=0.001)
LONG_128K = DecodeSpec("long-context GQA decode (4 seqs x 131072, 64/8 heads, d128)", 4,
                       4, 64, 8, 128, lens=(131072,) * 4)

DECODE_SPECS = {"tiny": TINY, "mha7b": MHA_7B, "gqa70b": GQA_70B, "long128k": LONG_128K}


def make_decode_workload(spec: DecodeSpec, device="cpu", gen_device=None,
                         lens_override: Optional[Sequence[int]] = None,
                         num_seqs_override: Optional[int] = None) -> DecodeWorkload:
    """Draw the inputs of one decode step for ``spec`` onto ``device``.

    ``lens_override`` / ``num_seqs_override`` shrink a spec (same head shape
    and value recipe) to sizes the oracle finishes quickly."""
    base = 1000 * spec.config_id
    S = num_seqs_override or spec.num_seqs
    if lens_override is not None:
        lens = [int(x) for x in lens_override]
        S = len(lens)
    elif spec.lens is not None:
        lens = list(spec.lens)[:S]
    else:
        lo, hi = spec.len_range
        lens = torch.randint(lo, hi + 1, (S,), generator=_cpu_gen(base + 5)).tolist()
    need = sum(blocks_for(L) for L in lens)
    nb = spec.num_blocks if (spec.num_blocks and lens_override is None) else max(
        1, math.ceil(1.25 * need))
    perm = torch.randperm(nb, generator=_cpu_gen(base + 6))
    tables, _ = build_block_tables(lens, perm)
    Hq, Hkv, d = spec.q_heads, spec.kv_heads, spec.d_head
    row_scale = None
    if spec.outlier_frac > 0:
        nrows = nb * BLOCK_SIZE * Hkv
        nout = int(round(spec.outlier_frac * nrows))
        sel = torch.randperm(nrows, generator=_cpu_gen(base + 7))[:nout]
        row_scale = (sel, spec.outlier_scale, d)
    pool_shape = (nb, BLOCK_SIZE, Hkv, d)
    k_cache = _randn_bf16(pool_shape, base + 1, device, gen_device, row_scale=row_scale)
    v_cache = _randn_bf16(pool_shape, base + 2, device, gen_device)
    q = _randn_bf16((S, Hq, d), base + 0, device, gen_device)
    k_new = _randn_bf16((S, Hkv, d), base + 3, device, gen_device)
    v_new = _randn_bf16((S, Hkv, d), base + 4, device, gen_device)
    slots = append_slots(tables, [[L - 1] for L in lens])
    scale = spec.scale if spec.scale is not None else 1.0 / math.sqrt(d)
    return DecodeWorkload(
        name=spec.name, q=q, k_cache=k_cache, v_cache=v_cache, k_new=k_new, v_new=v_new,
        slot_mapping=slots.to(device), block_tables=tables.to(device),
        context_lens=torch.tensor(lens, dtype=torch.int32, device=device), scale=float(scale),
        meta={"config_id": spec.config_id, "num_blocks": nb, "lens": lens})


# ---------------------------------------------------------------------------
# Continuous-batching mixed step: prefill chunks + decodes sharing a prefix.
# ---------------------------------------------------------------------------
@dataclass
class MixedWorkload:
    name: str
    k_cache: torch.Tensor         # [NB, bs, Hkv, d] bf16 (before the append)
    v_cache: torch.Tensor
    k_new: torch.Tensor           # [T_new, Hkv, d]: prefill chunk rows, then decode rows
    v_new: torch.Tensor
    slot_mapping: torch.Tensor    # [T_new] int64
    q_prefill: torch.Tensor       # [sum n, Hq, d] bf16 (packed chunks)
    q_start: torch.Tensor         # [P+1] int32
    prefill_tables: torch.Tensor  # [P, max_blocks] int32
    prefill_lens: torch.Tensor    # [P] int32 (prior + chunk)
    q_decode: torch.Tensor        # [D, Hq, d] bf16
    decode_tables: torch.Tensor   # [D, max_blocks] int32
    decode_lens: torch.Tensor     # [D] int32
    scale: float
    meta: dict = field(default_factory=dict)


@dataclass(frozen=True)
class MixedSpec:
    name: str
    config_id: int
    num_prefill: int
    chunk: int
    prior_range: tuple            # private prior context, inclusive uniform
    num_decode: int
    decode_median: float
    decode_sigma: float
    max_len: int
    shared_prefix: int            # tokens, a multiple of the block size
    q_heads: int
    kv_heads: int
    d_head: int


MIXED = MixedSpec("continuous-batching mixed step (8 prefill chunks x 512 + 248 decodes, "
                  "64/8 heads, d128, shared 1024-token prefix)", 5, 8, 512, (0, 4096), 248,
                  2048.0, 1.0, 32768, 1024, 64, 8, 128)


def _mixed_lengths(spec: MixedSpec, P: int, D: int, lo: int, hi: int, cap: int, prefix: int):
    """The priors of the P prefill sequences (prefix + U[lo, hi]) and the
    lengths of the D decode sequences, drawn in that order from one seeded
    generator."""
    g = _cpu_gen(1000 * spec.config_id + 5)
    priors = (prefix + torch.randint(lo, hi + 1, (P,), generator=g)).tolist()
    priv = torch.empty(D, dtype=torch.float64).log_normal_(
        math.log(spec.decode_median), spec.decode_sigma, generator=g)
    priv = torch.clamp(torch.round(priv), 1, max(1, cap - prefix)).to(torch.int64)
    return priors, (prefix + priv).tolist()


def mixed_prefill_priors(spec: MixedSpec = MIXED) -> list:
    """The tokens already cached for each prefill chunk of the mixed step
    (the same draw as make_mixed_workload), without building its pools."""
    return _mixed_lengths(spec, spec.num_prefill, spec.num_decode, *spec.prior_range,
                          spec.max_len, spec.shared_prefix)[0]


def make_mixed_workload(spec: MixedSpec = MIXED, device="cpu", gen_device=None,
                        num_prefill: Optional[int] = None, num_decode: Optional[int] = None,
                        chunk: Optional[int] = None, prior_range: Optional[tuple] = None,
                        decode_cap: Optional[int] = None, shared_prefix: Optional[int] = None
                        ) -> MixedWorkload:
    """Draw one mixed step.  Every sequence is [shared prefix] + private part;
    prefill sequences have prior = prefix + U[prior_range] and append a chunk;
    decode sequences have length prefix + round(LogNormal(ln median, sigma)),
    at least prefix + 1, at most the cap, and append their last token."""
    base = 1000 * spec.config_id
    P = spec.num_prefill if num_prefill is None else num_prefill
    D = spec.num_decode if num_decode is None else num_decode
    n = spec.chunk if chunk is None else chunk
    lo, hi = spec.prior_range if prior_range is None else prior_range
    cap = spec.max_len if decode_cap is None else decode_cap
    prefix = spec.shared_prefix if shared_prefix is None else shared_prefix
    if prefix % BLOCK_SIZE:
        raise ValueError("the shared prefix must fill whole blocks")
    priors, dlens = _mixed_lengths(spec, P, D, lo, hi, cap, prefix)
    plens = [p + n for p in priors]
    all_lens = plens + dlens
    pblocks = prefix // BLOCK_SIZE
    need = pblocks + sum(max(0, blocks_for(L) - pblocks) for L in all_lens)
    nb = max(1, math.ceil(1.25 * need))
    perm = torch.randperm(nb, generator=_cpu_gen(base + 6))
    tables, _ = build_block_tables(all_lens, perm, shared_prefix_blocks=pblocks)
    Hq, Hkv, d = spec.q_heads, spec.kv_heads, spec.d_head
    pool_shape = (nb, BLOCK_SIZE, Hkv, d)
    k_cache = _randn_bf16(pool_shape, base + 1, device, gen_device)
    v_cache = _randn_bf16(pool_shape, base + 2, device, gen_device)
    positions = [list(range(p, p + n)) for p in priors] + [[L - 1] for L in dlens]
    t_new = P * n + D
    k_new = _randn_bf16((t_new, Hkv, d), base + 3, device, gen_device)
    v_new = _randn_bf16((t_new, Hkv, d), base + 4, device, gen_device)
    slots = append_slots(tables, positions)
    q_all = _randn_bf16((P * n + D, Hq, d), base + 0, device, gen_device)
    q_start = torch.arange(P + 1, dtype=torch.int32) * n
    return MixedWorkload(
        name=spec.name, k_cache=k_cache, v_cache=v_cache, k_new=k_new, v_new=v_new,
        slot_mapping=slots.to(device), q_prefill=q_all[:P * n].contiguous(),
        q_start=q_start.to(device), prefill_tables=tables[:P].contiguous().to(device),
        prefill_lens=torch.tensor(plens, dtype=torch.int32, device=device),
        q_decode=q_all[P * n:].contiguous(), decode_tables=tables[P:].contiguous().to(device),
        decode_lens=torch.tensor(dlens, dtype=torch.int32, device=device),
        scale=1.0 / math.sqrt(d),
        meta={"config_id": spec.config_id, "num_blocks": nb, "prefill_lens": plens,
              "decode_lens": dlens, "chunk": n, "shared_prefix": prefix})


def bf16_bits(t: torch.Tensor):
    """Raw 16-bit patterns of a bf16 tensor as a numpy uint16 array (CPU)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")


def make_chunked_workload(q_heads: int, kv_heads: int, d_head: int, priors: Sequence[int],
                          chunks: Sequence[int], config_id: int = 6, shared_prefix: int = 0,
                          device="cpu", gen_device=None) -> MixedWorkload:
    """Prefill-only step with per-sequence chunk lengths: sequence s has
    ``priors[s]`` tokens already cached (the first ``shared_prefix`` of them in
    blocks common to every sequence) and appends ``chunks[s]`` new tokens."""
    base = 1000 * config_id
    if shared_prefix % BLOCK_SIZE:
        raise ValueError("the shared prefix must fill whole blocks")
    if any(p < shared_prefix for p in priors):
        raise ValueError("every prior must cover the shared prefix")
    lens = [int(p) + int(c) for p, c in zip(priors, chunks)]
    pblocks = shared_prefix // BLOCK_SIZE
    need = pblocks + sum(max(0, blocks_for(L) - pblocks) for L in lens)
    nb = max(1, math.ceil(1.25 * need))
    perm = torch.randperm(nb, generator=_cpu_gen(base + 6))
    tables, _ = build_block_tables(lens, perm, shared_prefix_blocks=pblocks)
    pool_shape = (nb, BLOCK_SIZE, kv_heads, d_head)
    k_cache = _randn_bf16(pool_shape, base + 1, device, gen_device)
    v_cache = _randn_bf16(pool_shape, base + 2, device, gen_device)
    positions = [list(range(int(p), int(p) + int(c))) for p, c in zip(priors, chunks)]
    t_new = sum(int(c) for c in chunks)
    k_new = _randn_bf16((t_new, kv_heads, d_head), base + 3, device, gen_device)
    v_new = _randn_bf16((t_new, kv_heads, d_head), base + 4, device, gen_device)
    q = _randn_bf16((t_new, q_heads, d_head), base + 0, device, gen_device)
    q_start = torch.zeros(len(chunks) + 1, dtype=torch.int32)
    q_start[1:] = torch.cumsum(torch.tensor([int(c) for c in chunks], dtype=torch.int32), 0)
    empty_tab = torch.zeros((0, tables.shape[1]), dtype=torch.int32)
    return MixedWorkload(
        name="chunked prefill", k_cache=k_cache, v_cache=v_cache, k_new=k_new, v_new=v_new,
        slot_mapping=append_slots(tables, positions).to(device), q_prefill=q,
        q_start=q_start.to(device), prefill_tables=tables.to(device),
        prefill_lens=torch.tensor(lens, dtype=torch.int32, device=device),
        q_decode=torch.empty((0, q_heads, d_head), dtype=torch.bfloat16, device=device),
        decode_tables=empty_tab.to(device),
        decode_lens=torch.empty(0, dtype=torch.int32, device=device),
        scale=1.0 / math.sqrt(d_head),
        meta={"config_id": config_id, "num_blocks": nb, "prefill_lens": lens, "decode_lens": [],
              "chunks": [int(c) for c in chunks], "shared_prefix": shared_prefix})


def fp8_pools(w, k_scale: float, v_scale: float):
    """Synthetic FP8 (e4m3) pools for a decode workload: the workload's bf16
    pool values over the per-pool scale, cast with torch's own float8_e4m3fn
    conversion (an independent library routine; the values are kept inside
    e4m3's range so no saturation is involved).  Returns uint8 code tensors."""
    out = []
    for pool, sc in ((w.k_cache, k_scale), (w.v_cache, v_scale)):
        x = pool.float() / float(sc)
        if float(x.abs().max()) >= 448.0:
            raise ValueError("scale too small for an in-range e4m3 pool")
        out.append(x.to(torch.float8_e4m3fn).view(torch.uint8).contiguous())
        del x
    return out[0], out[1]


# (k_scale, v_scale) per workload: powers of two that keep the pools in
# e4m3's range (the 70B-GQA K pool holds x100 outlier rows).
FP8_SCALES = {"gqa70b": (2.0, 0.03125), "mha7b": (0.03125, 0.03125),
              "long128k": (0.03125, 0.03125), "tiny": (0.03125, 0.03125)}
