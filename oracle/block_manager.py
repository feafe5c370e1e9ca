"""Oracle model of the host block manager of a paged KV cache (plain Python).

TEST INFRASTRUCTURE ONLY: used by ``tests/`` to check the native block
manager of the library operation by operation; never used by the product
path, and it shares no code with it.

What the pages describe, and what this model does:

* A pool of fixed-size blocks is allocated once at start; a sequence owns a
  list of physical block ids (its block table) and a block may sit anywhere in
  the pool ("Cache KV, attention et optimisation de l'inference", section
  "PagedAttention KV cache comme memoire virtuelle").  Finished sequences
  return their blocks to a free list (same page, exercise 3 of the section
  "Exercices").
* Prefix sharing by a chained hash: each full block carries a hash computed
  from the previous block's hash and its own token ids; a reference count
  keeps a shared block alive while any sequence uses it ("Maitriser les
  mecanismes cles de l'inference des grands modeles avec nano-vLLM", section
  "Implementation du cache").
* Copy-on-write: blocks of a common prompt are stored once and referenced by
  every request that shares them ("Cache KV, attention...", section
  "PageAtention"); a sequence that writes into a block it shares gets its own
  copy first.

Readings where the pages leave the policy open (the native manager follows
the same ones, so that both give identical block ids):

1. The hash of block ``j`` is FNV-1a (64-bit) continued from the hash of
   block ``j - 1`` over the ``4 * block_size`` little-endian bytes of the
   block's int32 token ids; the chain starts from the FNV offset basis.  A
   hash hit is accepted only if the cached block's token ids are equal too.
2. Only a leading run of full blocks is shared, and never the block holding
   the last prompt token, so at least one prompt token is always computed:
   at most ``(n - 1) // block_size`` blocks of an ``n``-token prompt hit.
3. The free list is first-in first-out, initially ``0 .. num_blocks - 1``.  A
   freed sequence returns its blocks last-to-first, so its head (the likely
   shared prefix) stays cached longest.  A block taken from the free list
   loses its cached hash; a cache hit on a free block takes it out of the
   list.
4. A block that becomes full by appends is hashed then; if the hash already
   names another block, the newest block takes the entry.
5. An operation that needs more free blocks than there are changes nothing
   and fails.
6. Copy-on-write happens in ``append_tokens`` (of at least one token) when
   the sequence's last block is partly filled and shared (reference count above one): a new block is
   taken, the pair (old, new) is reported for the caller to copy on the
   device, and the old block loses one reference.
"""

from __future__ import annotations

from collections import deque

FNV_OFFSET = 0xCBF29CE484222325
FNV_PRIME = 0x100000001B3
MASK64 = (1 << 64) - 1


class NoFreeBlocks(Exception):
    """The pool has fewer free blocks than the operation needs."""


def fnv1a64(data: bytes, h: int = FNV_OFFSET) -> int:
    """FNV-1a, 64-bit: for each byte, xor it in, then multiply by the prime."""
    for byte in data:
        h ^= byte
        h = (h * FNV_PRIME) & MASK64
    return h


def block_hash(prev: int, token_ids) -> int:
    data = b"".join(int(t).to_bytes(4, "little", signed=True) for t in token_ids)
    return fnv1a64(data, prev)


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks, self.bs = num_blocks, block_size
        self.ref = [0] * num_blocks
        self.hash = [None] * num_blocks        # cached hash of a full block
        self.content = [None] * num_blocks     # its token ids, to confirm a hit
        self.by_hash = {}
        self.free = deque(range(num_blocks))
        self.seqs = {}                         # id -> {"blocks", "tokens", "last_hash"}

    # ----------------------------------------------------------------- helpers
    def _take_free(self) -> int:
        b = self.free.popleft()
        h = self.hash[b]
        if h is not None:
            if self.by_hash.get(h) == b:
                del self.by_hash[h]
            self.hash[b] = None
            self.content[b] = None
        self.ref[b] = 1
        return b

    def _register(self, b: int, h: int, ids) -> None:
        self.hash[b] = h
        self.content[b] = tuple(ids)
        self.by_hash[h] = b

    # -------------------------------------------------------------- operations
    def add_sequence(self, seq_id: int, token_ids) -> int:
        """Blocks for a new prompt; returns the number of leading prompt
        tokens whose KV is already cached (shared blocks)."""
        if seq_id in self.seqs:
            raise KeyError(f"sequence {seq_id} exists")
        ids = list(token_ids)
        n, bs = len(ids), self.bs
        nblk = -(-n // bs)
        shareable = (n - 1) // bs if n > 0 else 0
        hashes, hits = [], []
        h = FNV_OFFSET
        for j in range(n // bs):
            h = block_hash(h, ids[j * bs:(j + 1) * bs])
            hashes.append(h)
        for j in range(shareable):
            b = self.by_hash.get(hashes[j])
            if b is None or self.content[b] != tuple(ids[j * bs:(j + 1) * bs]):
                break
            hits.append(b)
        need = (nblk - len(hits)) + sum(1 for b in hits if self.ref[b] == 0)
        if need > len(self.free):
            raise NoFreeBlocks(need)
        blocks = []
        for b in hits:
            if self.ref[b] == 0:
                self.free.remove(b)
            self.ref[b] += 1
            blocks.append(b)
        for j in range(len(hits), nblk):
            b = self._take_free()
            blocks.append(b)
            if j < len(hashes):
                self._register(b, hashes[j], ids[j * bs:(j + 1) * bs])
        self.seqs[seq_id] = {"blocks": blocks, "tokens": ids,
                             "last_hash": hashes[-1] if hashes else FNV_OFFSET}
        return len(hits) * bs

    def append_tokens(self, seq_id: int, token_ids):
        """Reserve slots for new tokens; returns (slots, copies) where copies
        are (src_block, dst_block) pairs to copy before the slots are written."""
        s = self.seqs[seq_id]
        ids = list(token_ids)
        n, bs, L = len(ids), self.bs, len(s["tokens"])
        blocks = s["blocks"]
        cow = n > 0 and L % bs != 0 and self.ref[blocks[-1]] > 1
        need = int(cow) + (-(-(L + n) // bs) - (-(-L // bs)))
        if need > len(self.free):
            raise NoFreeBlocks(need)
        copies = []
        if cow:
            old = blocks[-1]
            new = self._take_free()
            self.ref[old] -= 1
            blocks[-1] = new
            copies.append((old, new))
        slots = []
        for i in range(n):
            pos = L + i
            if pos % bs == 0:
                blocks.append(self._take_free())
            slots.append(blocks[pos // bs] * bs + pos % bs)
        s["tokens"].extend(ids)
        for j in range(L // bs, (L + n) // bs):
            chunk = s["tokens"][j * bs:(j + 1) * bs]
            s["last_hash"] = block_hash(s["last_hash"], chunk)
            self._register(blocks[j], s["last_hash"], chunk)
        return slots, copies

    def fork(self, parent: int, child: int) -> None:
        if child in self.seqs:
            raise KeyError(f"sequence {child} exists")
        p = self.seqs[parent]
        for b in p["blocks"]:
            self.ref[b] += 1
        self.seqs[child] = {"blocks": list(p["blocks"]), "tokens": list(p["tokens"]),
                            "last_hash": p["last_hash"]}

    def free_sequence(self, seq_id: int) -> None:
        s = self.seqs.pop(seq_id)
        for b in reversed(s["blocks"]):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.append(b)

    # ------------------------------------------------------------------ queries
    def block_table(self, seq_id: int):
        return list(self.seqs[seq_id]["blocks"])

    def seq_len(self, seq_id: int) -> int:
        return len(self.seqs[seq_id]["tokens"])

    def num_free_blocks(self) -> int:
        return len(self.free)

    def refcount(self, b: int) -> int:
        return self.ref[b]

    def slots(self, seq_id: int, start: int, count: int):
        blocks, bs = self.seqs[seq_id]["blocks"], self.bs
        return [blocks[p // bs] * bs + p % bs for p in range(start, start + count)]


def copy_blocks(k_cache, v_cache, pairs):
    """The device side of copy-on-write: block ``dst`` of both pools becomes a
    copy of block ``src`` for every (src, dst) pair (numpy arrays, in place).
    No destination may also be a source or appear twice, so the order in
    which the pairs are applied does not matter."""
    for src, dst in pairs:
        k_cache[dst] = k_cache[src]
        v_cache[dst] = v_cache[src]


def num_blocks_for_budget(usable_bytes, model_bytes, activation_peak_bytes, num_layers,
                          block_size, kv_heads, d_head, dtype_size):
    """Pool size from a memory budget, as the nano-vLLM page sizes it
    (section "Implementation du cache"): what is left after the weights and
    the activation peak, divided by the bytes of one block over all layers
    (K and V, ``block_size`` tokens, the KV heads held by this rank)."""
    per_block = 2 * int(num_layers) * int(block_size) * int(kv_heads) * int(d_head) * int(dtype_size)
    left = int(usable_bytes) - int(model_bytes) - int(activation_peak_bytes)
    return max(0, left // per_block)
