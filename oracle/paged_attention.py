"""Oracle for attention over a paged KV cache (numpy, float64).

TEST INFRASTRUCTURE ONLY: used by ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU baseline, never by the product path.  Shares no code with
the CUDA library.

What the method computes, and where the pages define it:

* KV append -- "Maitriser les mecanismes cles de l'inference des grands modeles
  avec nano-vLLM", section "Ecriture dans le cache": each new token ``t`` with
  ``slot_mapping[t] != -1`` has its K and V rows copied into the cache row
  ``slot``; a slot is ``physical_block * block_size + offset`` and ``-1`` means
  "skip this token".
* Paging -- "Cache KV, attention et optimisation de l'inference", section
  "PagedAttention KV cache comme memoire virtuelle" (16-token blocks, a page
  table maps logical block positions to physical blocks), and the nano-vLLM
  page, section "Cache KV" (a mapping table turns continuous logical addresses
  into scattered physical ones).  The pool of one layer is
  ``[num_blocks, block_size, kv_heads, d_head]`` (nano-vLLM page, section
  "Implementation du cache").
* Attention -- "Optimisation de l'inference", section "Etape 2: Attention avec
  KV Cache": ``softmax(q K^T / sqrt(d) + mask) V`` where, for more than one
  query, the mask is upper-triangular with offset ``Tk - Tq + 1`` (a
  bottom-right aligned causal mask).  Decode is the single-query case; the
  cache is updated first and the new token attends over the whole cache
  including itself (section "Etape 1", ``update`` returns ``[:end]``).
* GQA -- "第 10 讲：推理（Inference）", "核心概念与定义": N query heads share K
  key/value heads.  Reading (the pages do not fix the mapping): query head
  ``h`` uses KV head ``h // (N/K)``.
* Online softmax -- "Cache KV, attention et optimisation de l'inference",
  section "Etape 2: softmax en carreaux": running max and running sum, the old
  accumulator rescaled by ``exp(m_old - m_new)``, division by the sum at the
  end.
* Split-K merge -- the CS336 page only names FlashDecoding; the plain reading
  used here: each partition returns its normalised output and its
  log-sum-exp, and the partitions are combined with weights
  ``exp(lse_p - max_p lse_p)``.
* KV bytes -- "Optimisation de l'inference", section "Cache KV" (memory
  formula) and "Cache KV, attention et optimisation de l'inference", section
  "Mathematiques de cache KV": ``2 * kv_heads * head_dim * dtype_size`` bytes
  per token per layer.

Readings where the pages are silent: ``context_lens`` include the tokens
appended in the same step; a sequence with ``context_len == 0`` yields zeros;
the causal mask is exact exclusion (the pages add ``-1e9``, which has the same
effect in float64); the scale is the float32 value the kernels receive,
widened to float64.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_bits_to_f64",
    "f64_to_bf16_bits",
    "kv_append",
    "gather_sequence_kv",
    "attention",
    "paged_decode_attention",
    "paged_prefill_attention",
    "online_softmax_attention",
    "split_partials",
    "merge_partials",
    "kv_bytes_per_token_per_layer",
    "kv_bytes_per_token",
    "kv_cache_bytes",
]


# ---------------------------------------------------------------------------
# bf16 <-> float64.  bf16 is the upper 16 bits of an IEEE binary32 value, so
# widening is exact: shift the pattern into the high half of a uint32 and
# reinterpret it.
# ---------------------------------------------------------------------------
def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    bits = np.asarray(bits)
    if bits.dtype != np.uint16:
        raise TypeError(f"expected uint16 bf16 bit patterns, got {bits.dtype}")
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 bit patterns (via binary32, nearest-even).

    Used only to build test inputs; the double rounding through binary32 is
    not correctly rounded from binary64 in every case, which does not matter
    for that purpose.
    """
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return rounded.astype(np.uint16)


def _as_f64(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return bf16_bits_to_f64(x)
    return x.astype(np.float64)


# ---------------------------------------------------------------------------
# KV append (nano-vLLM page, "Ecriture dans le cache")
# ---------------------------------------------------------------------------
def kv_append(k_new, v_new, slot_mapping, k_cache, v_cache):
    """Scatter new K/V rows into copies of the caches.

    k_new, v_new: ``[T, kv_heads, d]`` (any dtype; bf16 as uint16 patterns)
    slot_mapping: ``[T]`` integers, ``slot = block * block_size + offset`` or -1
    k_cache, v_cache: ``[num_blocks, block_size, kv_heads, d]``, same dtype

    Returns new ``(k_cache, v_cache)`` arrays; the inputs are not modified.
    The copy is a bit copy, so the result is exact for any dtype.
    """
    k_new = np.asarray(k_new)
    v_new = np.asarray(v_new)
    slots = np.asarray(slot_mapping).astype(np.int64)
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    num_blocks, block_size = kc.shape[0], kc.shape[1]
    if k_new.shape[0] != slots.shape[0] or v_new.shape[0] != slots.shape[0]:
        raise ValueError("k_new, v_new and slot_mapping disagree on the token count")
    if k_new.shape[1:] != kc.shape[2:] or v_new.shape[1:] != vc.shape[2:]:
        raise ValueError("token rows do not match the cache row shape")
    for t in range(slots.shape[0]):
        slot = int(slots[t])
        if slot == -1:
            continue
        if slot < 0 or slot >= num_blocks * block_size:
            raise ValueError(f"slot {slot} of token {t} is outside the pool")
        kc[slot // block_size, slot % block_size] = k_new[t]
        vc[slot // block_size, slot % block_size] = v_new[t]
    return kc, vc


def kv_append_checked(k_new, v_new, slot_mapping, k_cache, v_cache):
    """The append with repeated slots rejected.

    The nano-vLLM page's slot mapping ("Ecriture dans le cache") gives every
    new token its own cache row; two tokens naming one row would leave that
    row undefined.  Reading: such a mapping is rejected as a whole.  Returns
    ``(k_cache, v_cache, rejected)``: unchanged copies and True when a slot
    other than -1 appears twice, else ``kv_append``'s result and False.
    """
    slots = np.asarray(slot_mapping).astype(np.int64)
    seen = set()
    for slot in slots.tolist():
        if slot == -1:
            continue
        if slot in seen:
            return np.array(k_cache, copy=True), np.array(v_cache, copy=True), True
        seen.add(slot)
    kc, vc = kv_append(k_new, v_new, slots, k_cache, v_cache)
    return kc, vc, False


# ---------------------------------------------------------------------------
# Paging: logical position j of a sequence lives in block_table[j // bs], row
# j % bs (page table of the PagedAttention sections).
# ---------------------------------------------------------------------------
def gather_sequence_kv(cache, block_table, length):
    """Contiguous ``[length, kv_heads, d]`` rows of one sequence (cache dtype)."""
    cache = np.asarray(cache)
    num_blocks, block_size = cache.shape[0], cache.shape[1]
    length = int(length)
    if length < 0:
        raise ValueError("negative context length")
    nblk = -(-length // block_size)
    table = np.asarray(block_table).astype(np.int64)[:nblk]
    if table.shape[0] < nblk:
        raise ValueError("block table shorter than the context needs")
    if nblk and (table.min() < 0 or table.max() >= num_blocks):
        raise ValueError("block id outside the pool")
    rows = cache[table].reshape((nblk * block_size,) + cache.shape[2:])
    return rows[:length]


# ---------------------------------------------------------------------------
# Attention ("Optimisation de l'inference", "Etape 2: Attention avec KV Cache")
# ---------------------------------------------------------------------------
def attention(q, k, v, scale, causal):
    """softmax(q k^T * scale [+ bottom-right causal mask]) v, per query head.

    q: ``[n, q_heads, d]``; k, v: ``[L, kv_heads, d]`` -- the n queries are the
    last n positions of the L keys.  Returns ``[n, q_heads, d_v]`` float64.
    """
    q = _as_f64(q)
    k = _as_f64(k)
    v = _as_f64(v)
    n, q_heads, _ = q.shape
    length, kv_heads, _ = k.shape
    if q_heads % kv_heads:
        raise ValueError("q_heads must be a multiple of kv_heads")
    group = q_heads // kv_heads
    out = np.zeros((n, q_heads, v.shape[2]), dtype=np.float64)
    if n == 0 or length == 0:
        return out
    if causal and n > length:
        raise ValueError("a causal chunk cannot be longer than its context")
    sc = float(np.float32(scale))
    key_pos = np.arange(length)
    query_pos = length - n + np.arange(n)
    for h in range(q_heads):
        kvh = h // group
        s = (q[:, h, :] @ k[:, kvh, :].T) * sc
        if causal:
            s = np.where(key_pos[None, :] <= query_pos[:, None], s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        p /= p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ v[:, kvh, :]
    return out


def paged_decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale):
    """One query per sequence over its paged history (including itself).

    q: ``[S, q_heads, d]``; caches ``[num_blocks, bs, kv_heads, d]``;
    block_tables ``[S, max_blocks]``; context_lens ``[S]``.
    Returns ``[S, q_heads, d]`` float64.
    """
    q = np.asarray(q)
    lens = np.asarray(context_lens).astype(np.int64)
    tables = np.asarray(block_tables)
    out = np.zeros(q.shape, dtype=np.float64)
    for s in range(q.shape[0]):
        kk = gather_sequence_kv(k_cache, tables[s], lens[s])
        vv = gather_sequence_kv(v_cache, tables[s], lens[s])
        out[s] = attention(q[s:s + 1], kk, vv, scale, causal=False)[0]
    return out


def paged_prefill_attention(q, q_start, k_cache, v_cache, block_tables, context_lens,
                            causal, scale):
    """Chunked prefill: the rows ``q_start[s]:q_start[s+1]`` of the packed
    ``q [total, q_heads, d]`` are the last tokens of sequence s, whose context
    (``context_lens[s]``) already holds their K/V.  Returns ``[total, q_heads, d]``.
    """
    q = np.asarray(q)
    starts = np.asarray(q_start).astype(np.int64)
    lens = np.asarray(context_lens).astype(np.int64)
    tables = np.asarray(block_tables)
    out = np.zeros(q.shape, dtype=np.float64)
    for s in range(starts.shape[0] - 1):
        a, b = int(starts[s]), int(starts[s + 1])
        if b < a:
            raise ValueError("q_start must be non-decreasing")
        kk = gather_sequence_kv(k_cache, tables[s], lens[s])
        vv = gather_sequence_kv(v_cache, tables[s], lens[s])
        out[a:b] = attention(q[a:b], kk, vv, scale, causal=bool(causal))
    return out


# ---------------------------------------------------------------------------
# Online (tiled) softmax ("Cache KV, attention et optimisation de l'inference",
# "Etape 2: softmax en carreaux"), for one query row and one head at a time.
# ---------------------------------------------------------------------------
def online_softmax_attention(q, k, v, scale, tile, causal=False):
    """Same result as ``attention`` computed tile by tile with a running max
    and a running sum; the old accumulator is rescaled by exp(m_old - m_new)."""
    q = _as_f64(q)
    k = _as_f64(k)
    v = _as_f64(v)
    n, q_heads, _ = q.shape
    length, kv_heads, _ = k.shape
    group = q_heads // kv_heads
    sc = float(np.float32(scale))
    out = np.zeros((n, q_heads, v.shape[2]), dtype=np.float64)
    for i in range(n):
        visible = length - n + i + 1 if causal else length
        for h in range(q_heads):
            kvh = h // group
            m = -np.inf
            ssum = 0.0
            acc = np.zeros(v.shape[2], dtype=np.float64)
            for start in range(0, visible, tile):
                stop = min(start + tile, visible)
                scores = (k[start:stop, kvh, :] @ q[i, h, :]) * sc
                new_m = max(m, float(scores.max()))
                exp_old = np.exp(m - new_m) if m != -np.inf else 0.0
                exp_new = np.exp(scores - new_m)
                ssum = ssum * exp_old + float(exp_new.sum())
                acc = acc * exp_old + exp_new @ v[start:stop, kvh, :]
                m = new_m
            if visible > 0:
                out[i, h] = acc / ssum
    return out


# ---------------------------------------------------------------------------
# Split-K partitions and their log-sum-exp merge (FlashDecoding, named on the
# CS336 page; the merge is the plain reading stated in the module docstring).
# ---------------------------------------------------------------------------
def split_partials(q, k, v, scale, part_tokens):
    """Per partition p covering keys [p*C, min(L, (p+1)*C)): the normalised
    output ``o_p [q_heads, d]`` and ``lse_p [q_heads]`` (natural log of the
    partition's sum of exp(score)).  q is one query ``[q_heads, d]``."""
    q = _as_f64(q)
    k = _as_f64(k)
    v = _as_f64(v)
    length, kv_heads, _ = k.shape
    q_heads = q.shape[0]
    group = q_heads // kv_heads
    sc = float(np.float32(scale))
    parts = []
    for start in range(0, length, part_tokens):
        stop = min(start + part_tokens, length)
        o = np.zeros((q_heads, v.shape[2]), dtype=np.float64)
        lse = np.zeros(q_heads, dtype=np.float64)
        for h in range(q_heads):
            kvh = h // group
            s = (k[start:stop, kvh, :] @ q[h]) * sc
            m = s.max()
            e = np.exp(s - m)
            o[h] = (e @ v[start:stop, kvh, :]) / e.sum()
            lse[h] = m + np.log(e.sum())
        parts.append((o, lse))
    return parts


def merge_partials(parts):
    """out = sum_p exp(lse_p - M) o_p / sum_p exp(lse_p - M), M = max_p lse_p."""
    lses = np.stack([lse for _, lse in parts])          # [P, q_heads]
    outs = np.stack([o for o, _ in parts])              # [P, q_heads, d]
    big = lses.max(axis=0)
    w = np.exp(lses - big[None, :])
    return (w[:, :, None] * outs).sum(axis=0) / w.sum(axis=0)[:, None]


# ---------------------------------------------------------------------------
# KV byte counts ("Optimisation de l'inference", "Cache KV" memory formula;
# "Cache KV, attention et optimisation de l'inference", "Mathematiques de
# cache KV"; nano-vLLM page, "Implementation du cache" pool tensor).
# ---------------------------------------------------------------------------
def kv_bytes_per_token_per_layer(kv_heads, d_head, dtype_size):
    """K and V rows of one token in one layer: 2 * kv_heads * d_head * size."""
    return 2 * int(kv_heads) * int(d_head) * int(dtype_size)


def kv_bytes_per_token(num_layers, kv_heads, d_head, dtype_size):
    """Whole-model KV bytes per token: layers times the per-layer figure."""
    return int(num_layers) * kv_bytes_per_token_per_layer(kv_heads, d_head, dtype_size)


def kv_cache_bytes(num_blocks, block_size, kv_heads, d_head, dtype_size):
    """Bytes of one layer's K and V pools ``2 x [num_blocks, bs, kv_heads, d]``."""
    return 2 * int(num_blocks) * int(block_size) * int(kv_heads) * int(d_head) * int(dtype_size)
