"""The library's native block manager against the oracle model, operation by
operation (no GPU needed): identical cached-token counts, slots, copy pairs,
block tables, reference counts and free-list order, and the same refusals."""

import random

import pytest

import oracle
from oracle.block_manager import BlockManager as OracleBM, NoFreeBlocks as OracleNoFree

BS = 16


@pytest.fixture(scope="module")
def pk():
    import os
    from paged_kv_cache_52_gb300 import build as b
    if not os.path.exists(b.LIB_PATH):
        b.build()
    from paged_kv_cache_52_gb300 import pagedkv
    return pagedkv


def _state(bm, live, num_blocks, native):
    tables = {s: bm.block_table(s) for s in sorted(live)}
    lens = {s: bm.seq_len(s) for s in sorted(live)}
    refs = [bm.refcount(b) for b in range(num_blocks)]
    free = bm.free_list() if native else list(bm.free)
    return tables, lens, refs, free, bm.num_free_blocks()


def _run_both(pk, seed, steps, num_blocks, vocab=40, max_prompt=90):
    rng = random.Random(seed)
    nat, ref = pk.BlockManager(num_blocks, BS), OracleBM(num_blocks, BS)
    bases = [[rng.randrange(vocab) for _ in range(max_prompt)] for _ in range(4)]
    live, next_id = set(), 0
    counts = {"add": 0, "hit": 0, "cow": 0, "full": 0}
    for _ in range(steps):
        op = rng.random()
        if op < 0.3 or not live:
            base = rng.choice(bases)
            toks = base[:rng.randrange(0, max_prompt)] + [rng.randrange(vocab)
                                                          for _ in range(rng.randrange(0, 20))]
            sid, call = next_id, ("add_sequence", next_id, toks)
            next_id += 1
        elif op < 0.7:
            sid = rng.choice(sorted(live))
            call = ("append_tokens", sid, [rng.randrange(vocab) for _ in range(rng.randrange(0, 24))])
        elif op < 0.85:
            sid = next_id
            call = ("fork", rng.choice(sorted(live)), next_id)
            next_id += 1
        else:
            sid = rng.choice(sorted(live))
            call = ("free_sequence", sid)
        name, *args = call
        try:
            want = getattr(ref, name)(*args)
            want_err = None
        except OracleNoFree:
            want, want_err = None, "full"
        try:
            got = getattr(nat, name)(*args)
            got_err = None
        except pk.NoFreeBlocks:
            got, got_err = None, "full"
        assert (got_err, got) == (want_err, want), (seed, call)
        if want_err:
            counts["full"] += 1
        elif name == "add_sequence":
            live.add(sid)
            counts["add"] += 1
            counts["hit"] += want > 0
        elif name == "fork":
            live.add(sid)
        elif name == "free_sequence":
            live.discard(sid)
        elif want[1]:
            counts["cow"] += 1
        assert _state(nat, live, num_blocks, True) == _state(ref, live, num_blocks, False), (seed, call)
    if live:
        S = len(live)
        ids = sorted(live)
        mb = max(len(ref.block_table(s)) for s in ids) + 1
        tables, lens = nat.block_tables(ids, mb)
        for r, s in enumerate(ids):
            row = ref.block_table(s)
            assert tables[r, :len(row)].tolist() == row and not tables[r, len(row):].any()
            assert int(lens[r]) == ref.seq_len(s)
        assert tables.shape == (S, mb)
    nat.close()
    return counts


@pytest.mark.parametrize("seed,num_blocks", [(0, 40), (1, 64), (2, 24), (3, 200)])
def test_native_matches_oracle_operation_by_operation(pk, seed, num_blocks):
    c = _run_both(pk, seed, steps=600, num_blocks=num_blocks)
    assert c["add"] > 0 and c["hit"] > 0 and c["cow"] > 0
    if num_blocks <= 40:
        assert c["full"] > 0          # the small pools do run out


def test_native_refusals(pk):
    bm = pk.BlockManager(3, BS)
    with pytest.raises(pk.PagedKVError):
        pk.BlockManager(0, BS)
    assert bm.add_sequence(1, range(40)) == 0
    with pytest.raises(pk.PagedKVError) as e:
        bm.add_sequence(1, [1])                          # id already registered
    assert e.value.status == -1
    with pytest.raises(pk.NoFreeBlocks):
        bm.add_sequence(2, range(100, 117))
    assert bm.free_list() == [] and bm.block_table(1) == [0, 1, 2]
    bm.fork(1, 2)
    with pytest.raises(pk.NoFreeBlocks):
        bm.append_tokens(2, [1])                          # the copy-on-write block
    assert bm.refcount(2) == 2 and bm.seq_len(2) == 40
    for bad in (lambda: bm.fork(9, 10), lambda: bm.free_sequence(9), lambda: bm.slots(1, 30, 11),
                lambda: bm.seq_len(9), lambda: bm.block_tables([1, 2], 2)):
        with pytest.raises(pk.PagedKVError):
            bad()
    assert bm.refcount(-1) == -1 and bm.refcount(3) == -1
    bm.close()
    # a copy-on-write append with no room for the pair is refused and changes nothing
    import ctypes
    bm = pk.BlockManager(8, BS)
    bm.add_sequence(1, range(20))
    bm.fork(1, 2)
    before = (bm.free_list(), bm.refcount(1), bm.seq_len(2), bm.block_table(2))
    n = ctypes.c_int32()
    st = pk.lib.pkv_bm_append_tokens(bm._h, 2, (ctypes.c_int32 * 1)(5), 1, (ctypes.c_int64 * 1)(),
                                     None, 0, ctypes.byref(n))
    assert st == -1
    assert (bm.free_list(), bm.refcount(1), bm.seq_len(2), bm.block_table(2)) == before
    bm.close()


def test_pool_size_matches_oracle(pk):
    gib = 1 << 30
    for args in [(100 * gib, 40 * gib, 5 * gib, 80, BS, 8, 128, 2),
                 (280 * gib, 140 * gib, 8 * gib, 80, BS, 1, 128, 2),     # 8-way split KV heads
                 (280 * gib, 16 * gib, 4 * gib, 32, BS, 32, 128, 1),     # FP8 pool
                 (gib, 2 * gib, 0, 80, BS, 8, 128, 2)]:
        assert pk.blocks_for_budget(*args) == oracle.num_blocks_for_budget(*args)
    with pytest.raises(ValueError):
        pk.blocks_for_budget(gib, 0, 0, 0, BS, 8, 128, 2)
