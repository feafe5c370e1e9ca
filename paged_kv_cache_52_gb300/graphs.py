"""CUDA-graph replay of the decode step with batch-size buckets.

The nano-vLLM page ("Maitriser les mecanismes cles de l'inference des grands
modeles avec nano-vLLM", section "CUDA Graph") captures the decode step once
per batch-size bucket and pads each live batch to the smallest bucket that
holds it, so a step costs one graph launch instead of one launch per kernel.

Here a step is the library's decode step -- ``paged_decode_step``: each
sequence's new token appended, then attended, the append's kernel running
beside the attention -- captured on static buffers.  Padding needs no special case in the kernels: a padded sequence has
``context_len == 0`` (its output is zero) and slot ``-1`` (nothing is
appended).  The split-K workspace is allocated once per bucket before
capture, so the captured calls allocate nothing.  This module only stages
inputs and replays graphs; every step of the computation runs in the
library's kernels.
"""

from __future__ import annotations

import bisect
from typing import Dict, Optional, Sequence

import torch

from . import pagedkv

DEFAULT_BUCKETS = (1, 2, 4, 8, 16, 32, 64, 128, 256)


class _Bucket:
    def __init__(self, size, q_heads, kv_heads, d_head, max_blocks, max_context_len, device):
        self.size = size
        self.q = torch.zeros(size, q_heads, d_head, dtype=torch.bfloat16, device=device)
        self.k_new = torch.zeros(size, kv_heads, d_head, dtype=torch.bfloat16, device=device)
        self.v_new = torch.zeros_like(self.k_new)
        self.slots = torch.full((size,), -1, dtype=torch.int64, device=device)
        self.tables = torch.zeros(size, max_blocks, dtype=torch.int32, device=device)
        self.lens = torch.zeros(size, dtype=torch.int32, device=device)
        self.out = torch.zeros(size, q_heads, d_head, dtype=torch.float32, device=device)
        self.workspace = pagedkv.decode_workspace(size, q_heads, kv_heads, d_head,
                                                  max_context_len, device)
        self.graph: Optional[torch.cuda.CUDAGraph] = None


class DecodeGraphRunner:
    """Captures append + decode once per bucket over fixed KV pools and
    replays the graph of the smallest bucket that holds each batch."""

    def __init__(self, k_cache: torch.Tensor, v_cache: torch.Tensor, q_heads: int,
                 max_blocks_per_seq: int, max_context_len: int, scale: float,
                 buckets: Sequence[int] = DEFAULT_BUCKETS):
        self.k_cache, self.v_cache = k_cache, v_cache
        self.q_heads = q_heads
        self.kv_heads, self.d_head = k_cache.shape[2], k_cache.shape[3]
        self.max_blocks = max_blocks_per_seq
        self.max_context_len = max_context_len
        self.scale = scale
        self.sizes = sorted(set(int(b) for b in buckets))
        self.buckets: Dict[int, _Bucket] = {}

    def _step(self, b: _Bucket):
        pagedkv.paged_decode_step(b.q, b.k_new, b.v_new, b.slots, self.k_cache, self.v_cache,
                                  b.tables, b.lens, self.scale, out=b.out,
                                  max_context_len=self.max_context_len, workspace=b.workspace)

    def capture(self, size: int) -> _Bucket:
        b = _Bucket(size, self.q_heads, self.kv_heads, self.d_head, self.max_blocks,
                    self.max_context_len, self.k_cache.device)
        # one eager call first: per-kernel attributes are set outside capture
        side = torch.cuda.Stream(device=self.k_cache.device)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self._step(b)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self._step(b)
        b.graph = g
        self.buckets[size] = b
        return b

    def bucket_for(self, n: int) -> int:
        i = bisect.bisect_left(self.sizes, n)
        if i == len(self.sizes):
            raise ValueError(f"batch of {n} exceeds the largest bucket {self.sizes[-1]}")
        return self.sizes[i]

    def run(self, q, k_new, v_new, slot_mapping, block_tables, context_lens) -> torch.Tensor:
        """One decode step for a live batch of n sequences; returns out[:n]."""
        n = q.shape[0]
        size = self.bucket_for(n)
        b = self.buckets.get(size) or self.capture(size)
        b.q[:n].copy_(q)
        b.k_new[:n].copy_(k_new)
        b.v_new[:n].copy_(v_new)
        b.slots[:n].copy_(slot_mapping)
        b.slots[n:].fill_(-1)
        b.tables[:n, :block_tables.shape[1]].copy_(block_tables)
        b.lens[:n].copy_(context_lens)
        b.lens[n:].zero_()
        b.graph.replay()
        return b.out[:n]
