"""Pins of the oracle block manager against things other than itself: the
published FNV-1a test vectors, hand-worked sharing / copy-on-write cases, the
pool-size formula on the pages' own per-token figure, and a simulated cache
whose rows must always read back as each sequence's own history."""

import copy
import random

import numpy as np
import pytest

import oracle
from oracle.block_manager import BlockManager, NoFreeBlocks, FNV_OFFSET

BS = 16


def test_fnv1a64_published_vectors():
    # test vectors of the FNV specification (FNV-1a, 64-bit)
    assert oracle.fnv1a64(b"") == 0xCBF29CE484222325
    assert oracle.fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert oracle.fnv1a64(b"foobar") == 0x85944171F73967E8
    # chaining continues the same byte stream: hash(A) then B == hash(A + B)
    assert oracle.fnv1a64(b"bar", oracle.fnv1a64(b"foo")) == oracle.fnv1a64(b"foobar")
    assert oracle.block_hash(FNV_OFFSET, [1, -1]) == oracle.fnv1a64(
        b"\x01\x00\x00\x00\xff\xff\xff\xff")


def test_shared_prompt_is_stored_once():
    bm = BlockManager(8, BS)
    prompt = list(range(40))                      # 2 full blocks + 8 tokens
    assert bm.add_sequence(1, prompt) == 0
    assert bm.block_table(1) == [0, 1, 2]
    assert bm.add_sequence(2, prompt) == 32       # both full blocks shared
    assert bm.block_table(2) == [0, 1, 3]
    assert [bm.refcount(b) for b in range(4)] == [2, 2, 1, 1]
    assert bm.num_free_blocks() == 4
    # a different second block shares only the first
    other = prompt[:16] + [99] * 24
    assert bm.add_sequence(3, other) == 16
    assert bm.block_table(3)[0] == 0 and bm.refcount(0) == 3


def test_last_prompt_token_is_always_computed():
    bm = BlockManager(8, BS)
    p = list(range(32))                           # exactly two full blocks
    bm.add_sequence(1, p)
    assert bm.add_sequence(2, p) == 16            # block 1 holds the last token
    assert bm.add_sequence(3, p + [7]) == 32      # now it does not
    assert bm.add_sequence(4, [5]) == 0


def test_fork_then_append_copies_the_partial_block_once():
    bm = BlockManager(8, BS)
    bm.add_sequence(1, list(range(20)))           # blocks [0, 1], block 1 holds 4 tokens
    bm.fork(1, 2)
    assert bm.refcount(1) == 2
    slots, copies = bm.append_tokens(2, [100])
    assert copies == [(1, 2)] and slots == [2 * BS + 4]
    assert bm.block_table(2) == [0, 2] and bm.refcount(1) == 1
    slots, copies = bm.append_tokens(1, [200])    # block 1 is its own again
    assert copies == [] and slots == [1 * BS + 4]
    # a full shared last block needs no copy: the next token opens a new block
    bm2 = BlockManager(8, BS)
    bm2.add_sequence(1, list(range(16)))
    bm2.fork(1, 2)
    slots, copies = bm2.append_tokens(2, [1])
    assert copies == [] and slots == [1 * BS]
    # an empty append changes nothing
    bm2.fork(1, 3)
    assert bm2.append_tokens(3, []) == ([], [])


def test_exhaustion_changes_nothing():
    bm = BlockManager(3, BS)
    bm.add_sequence(1, list(range(40)))
    before = copy.deepcopy(bm.__dict__)
    with pytest.raises(NoFreeBlocks):
        bm.add_sequence(2, list(range(1000, 1017)))   # needs 2 blocks, 0 free
    assert bm.__dict__ == before
    bm.fork(1, 3)
    before = copy.deepcopy(bm.__dict__)
    with pytest.raises(NoFreeBlocks):
        bm.append_tokens(3, [1])                      # needs the copy-on-write block
    assert bm.__dict__ == before


def test_freed_blocks_stay_cached_until_reused():
    bm = BlockManager(4, BS)
    p = list(range(40))
    bm.add_sequence(1, p)
    bm.free_sequence(1)
    assert bm.num_free_blocks() == 4
    assert list(bm.free) == [3, 2, 1, 0]          # initial 3, then last-to-first
    assert bm.add_sequence(2, p) == 32            # hits on free blocks 0 and 1
    assert bm.block_table(2) == [0, 1, 3]
    bm.free_sequence(2)
    assert list(bm.free) == [2, 3, 1, 0]
    # new content takes blocks from the front of the free list
    assert bm.add_sequence(3, list(range(500, 564))) == 0
    assert bm.block_table(3) == [2, 3, 1, 0]      # evicts the cached prefix
    bm.free_sequence(3)
    assert bm.add_sequence(5, p) == 0             # prefix blocks were reused: no hit


def test_pool_size_formula():
    # per block over 80 layers, 8 KV heads, d 128, bf16: 16 tokens x the
    # 327,680 bytes per token the first page works out for a 70B model
    per_block = 2 * 80 * BS * 8 * 128 * 2
    assert per_block == 16 * 327_680
    gib = 1 << 30
    assert oracle.num_blocks_for_budget(100 * gib, 40 * gib, 5 * gib, 80, BS, 8, 128, 2) == 11264
    assert oracle.num_blocks_for_budget(gib, 2 * gib, 0, 80, BS, 8, 128, 2) == 0


# ------------------------------------------------------------------ simulation
def _row_value(prev: int, token: int) -> int:
    """Stand-in for a KV row: a value that depends on the whole prefix."""
    return (prev * 1_000_003 + token + 1) % ((1 << 61) - 1)


class _Sim:
    """A cache of one int64 'row' per slot, written only where the block
    manager says and read back through its block tables."""

    def __init__(self, bm, num_blocks):
        self.bm = bm
        self.cache = np.full((num_blocks, BS), -1, dtype=np.int64)
        self.truth = {}      # seq -> list of expected row values

    def _values(self, tokens, prev=0):
        out = []
        for t in tokens:
            prev = _row_value(prev, t)
            out.append(prev)
        return out

    def add(self, sid, tokens):
        cached = self.bm.add_sequence(sid, tokens)
        vals = self._values(tokens)
        for pos, slot in zip(range(cached, len(tokens)),
                             self.bm.slots(sid, cached, len(tokens) - cached)):
            self.cache.reshape(-1)[slot] = vals[pos]
        self.truth[sid] = vals
        return cached

    def append(self, sid, tokens):
        slots, copies = self.bm.append_tokens(sid, tokens)
        k = self.cache
        oracle.copy_blocks(k, k.copy(), copies)        # the V pool is not simulated
        prev = self.truth[sid][-1] if self.truth[sid] else 0
        vals = self._values(tokens, prev)
        for s, v in zip(slots, vals):
            self.cache.reshape(-1)[s] = v
        self.truth[sid] = self.truth[sid] + vals

    def fork(self, parent, child):
        self.bm.fork(parent, child)
        self.truth[child] = list(self.truth[parent])

    def free(self, sid):
        self.bm.free_sequence(sid)
        del self.truth[sid]

    def check(self):
        flat = self.cache.reshape(-1)
        for sid, vals in self.truth.items():
            slots = self.bm.slots(sid, 0, len(vals))
            assert flat[slots].tolist() == vals, f"sequence {sid} reads back wrong rows"
        counts = [0] * self.bm.num_blocks
        for sid in self.truth:
            for b in self.bm.block_table(sid):
                counts[b] += 1
        assert counts == [self.bm.refcount(b) for b in range(self.bm.num_blocks)]
        free = list(self.bm.free)
        assert len(set(free)) == len(free)
        assert sorted(free) == [b for b in range(self.bm.num_blocks) if counts[b] == 0]


def run_simulation(bm_cls, seed, steps=400, num_blocks=48):
    rng = random.Random(seed)
    sim = _Sim(bm_cls(num_blocks, BS), num_blocks)
    bases = [[rng.randrange(50) for _ in range(70)] for _ in range(3)]
    next_id, hits = 0, 0
    for _ in range(steps):
        live = list(sim.truth)
        op = rng.random()
        try:
            if op < 0.3 or not live:
                base = rng.choice(bases)
                tokens = base[:rng.randrange(0, 70)] + [rng.randrange(50)
                                                      for _ in range(rng.randrange(1, 20))]
                hits += sim.add(next_id, tokens) > 0
                next_id += 1
            elif op < 0.7:
                sim.append(rng.choice(live), [rng.randrange(50) for _ in range(rng.randrange(1, 20))])
            elif op < 0.85:
                sim.fork(rng.choice(live), next_id)
                next_id += 1
            else:
                sim.free(rng.choice(live))
        except NoFreeBlocks:
            pass
        sim.check()
    return hits


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_simulated_cache_reads_back_every_history(seed):
    assert run_simulation(BlockManager, seed) > 0     # prefix sharing did happen


class _NoCopyOnWrite(BlockManager):
    def append_tokens(self, seq_id, token_ids):
        blocks = self.seqs[seq_id]["blocks"]
        if not blocks:
            return super().append_tokens(seq_id, token_ids)
        last, saved = blocks[-1], self.ref[blocks[-1]]
        self.ref[last] = 1                            # pretend the block is not shared
        out = super().append_tokens(seq_id, token_ids)
        self.ref[last] += saved - 1                   # keep the counts themselves right
        return out


class _HitStaysFree(BlockManager):
    def add_sequence(self, seq_id, token_ids):
        free = list(self.free)
        cached = super().add_sequence(seq_id, token_ids)
        taken = [b for b in free if b not in self.free and self.ref[b] > 0
                 and b in self.seqs[seq_id]["blocks"][:cached // self.bs]]
        for b in taken:
            self.free.append(b)                       # forget to take the hit off the list
        return cached


@pytest.mark.parametrize("mutant", [_NoCopyOnWrite, _HitStaysFree])
def test_simulation_catches_planted_mistakes(mutant):
    with pytest.raises(AssertionError):
        for seed in range(6):
            run_simulation(mutant, seed)
