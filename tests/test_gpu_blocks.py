"""Copy-on-write block copies on the GPU are bit-exact against the oracle,
and a serving loop driven by the native block manager (shared prompt
prefixes, forks, copy-on-write, frees and cache hits on freed blocks) gives
attention outputs that match the oracle on each sequence's own contiguous
history."""

import numpy as np
import pytest
import torch

import oracle
from parity import assert_attention_close
from paged_kv_cache_52_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_52_gb300 import pagedkv
    pagedkv.get_device_error(clear=True)
    return pagedkv


def _pools(shape, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    if dtype == torch.uint8:
        k = torch.randint(0, 256, shape, generator=g, dtype=torch.uint8)
        v = torch.randint(0, 256, shape, generator=g, dtype=torch.uint8)
    else:
        k = torch.randn(shape, generator=g).to(dtype)
        v = torch.randn(shape, generator=g).to(dtype)
    return k, v


def _bits(t):
    return t.view(torch.uint8).numpy() if t.dtype == torch.uint8 else wl.bf16_bits(t)


def _copy_and_compare(pk, shape, dtype, pairs, seed):
    k0, v0 = _pools(shape, dtype, seed)
    kr, vr = _bits(k0).copy(), _bits(v0).copy()
    oracle.copy_blocks(kr, vr, pairs)
    kc, vc = k0.to(DEV), v0.to(DEV)
    pk.copy_blocks(kc, vc, torch.tensor(pairs, dtype=torch.int32, device=DEV).reshape(-1, 2))
    torch.cuda.synchronize()
    assert np.array_equal(_bits(kc.cpu()), kr)
    assert np.array_equal(_bits(vc.cpu()), vr)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.uint8])
def test_copy_blocks_bit_exact(pk, dtype):
    pairs = [(3, 17), (0, 5), (29, 1), (8, 9), (12, 30)]
    _copy_and_compare(pk, (40, 16, 8, 128), dtype, pairs, seed=11)
    assert pk.get_device_error(clear=True) == 0


def test_copy_blocks_many_pairs_strides_the_grid(pk):
    # 900 pairs = 1800 (pair, pool) items, more than one pass of the grid
    pairs = [(i, 1000 + i) for i in range(900)]
    _copy_and_compare(pk, (2000, 16, 2, 64), torch.bfloat16, pairs, seed=12)
    assert pk.get_device_error(clear=True) == 0


def test_copy_blocks_out_of_range_pair_is_skipped_and_reported(pk):
    k0, v0 = _pools((16, 16, 2, 64), torch.bfloat16, 13)
    kc, vc = k0.to(DEV), v0.to(DEV)
    pairs = torch.tensor([[1, 2], [0, 16], [-1, 3], [4, 5]], dtype=torch.int32, device=DEV)
    pk.copy_blocks(kc, vc, pairs)
    torch.cuda.synchronize()
    kr, vr = wl.bf16_bits(k0).copy(), wl.bf16_bits(v0).copy()
    oracle.copy_blocks(kr, vr, [(1, 2), (4, 5)])
    assert np.array_equal(wl.bf16_bits(kc.cpu()), kr)
    assert np.array_equal(wl.bf16_bits(vc.cpu()), vr)
    assert pk.get_device_error(clear=True) == 0x2
    pk.copy_blocks(kc, vc, torch.empty(0, 2, dtype=torch.int32, device=DEV))   # nothing to do


# ------------------------------------------------------------ serving loop
HKV, HQ, D, NB = 2, 8, 64, 96
SCALE = D ** -0.5


def _row_value(prev, token):
    return (prev * 1_000_003 + token + 1) % ((1 << 61) - 1)


class _Histories:
    """K/V rows that depend only on the token prefix, as a model's would:
    equal prefixes give equal rows, so sharing their blocks is exact."""

    def __init__(self):
        self.chain, self.k, self.v = {}, {}, {}

    def extend(self, sid, tokens, parent=None):
        if parent is not None:
            self.chain[sid] = list(self.chain[parent])
            self.k[sid], self.v[sid] = list(self.k[parent]), list(self.v[parent])
        self.chain.setdefault(sid, [])
        self.k.setdefault(sid, [])
        self.v.setdefault(sid, [])
        for t in tokens:
            r = _row_value(self.chain[sid][-1] if self.chain[sid] else 0, t)
            self.chain[sid].append(r)
            rows = np.random.default_rng(r).standard_normal((2, HKV, D)).astype(np.float32)
            bf = torch.from_numpy(rows).to(torch.bfloat16)
            self.k[sid].append(bf[0])
            self.v[sid].append(bf[1])

    def rows(self, sid, start=0, stop=None):
        k = torch.stack(self.k[sid][start:stop])
        v = torch.stack(self.v[sid][start:stop])
        return k, v


def _append_rows(pk, hist, items, kc, vc):
    """items: [(sid, start, stop, slots)] -> one kv_append for all rows."""
    ks, vs, slots = [], [], []
    for sid, a, b, sl in items:
        k, v = hist.rows(sid, a, b)
        ks.append(k)
        vs.append(v)
        slots.extend(sl)
    if not slots:
        return
    pk.kv_append(torch.cat(ks).to(DEV), torch.cat(vs).to(DEV),
                 torch.tensor(slots, dtype=torch.int64, device=DEV), kc, vc)


def _oracle(hist, sid, q, causal):
    k, v = hist.rows(sid)
    return oracle.attention(wl.bf16_bits(q), wl.bf16_bits(k), wl.bf16_bits(v), SCALE, causal)


def test_serving_loop_driven_by_the_block_manager(pk):
    g = torch.Generator().manual_seed(21)
    rnd = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)   # noqa: E731
    bm, hist = pk.BlockManager(NB), _Histories()
    kc = torch.full((NB, 16, HKV, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    vc = torch.full_like(kc, float("nan"))      # canary: a row never written reads NaN
    base = torch.randint(0, 50, (60,), generator=g).tolist()
    own = lambda n: torch.randint(50, 100, (n,), generator=g).tolist()   # noqa: E731
    live, stats = [], {"hits": 0, "copies": 0}

    def prefill(prompts):
        """Register prompts, append the rows of their uncached tail, and check
        the chunked prefill of that tail against the oracle."""
        items, chunks = [], []
        for sid, toks in prompts:
            cached = bm.add_sequence(sid, toks)
            stats["hits"] += cached > 0
            hist.extend(sid, toks)
            items.append((sid, cached, len(toks), bm.slots(sid, cached, len(toks) - cached)))
            chunks.append((sid, len(toks) - cached))
            live.append(sid)
        _append_rows(pk, hist, items, kc, vc)
        ids = [s for s, _ in chunks]
        mb = max(len(bm.block_table(s)) for s in ids)
        tables, lens = bm.block_tables(ids, mb)
        q = rnd(sum(n for _, n in chunks), HQ, D)
        starts = np.cumsum([0] + [n for _, n in chunks]).tolist()
        out = pk.paged_prefill_attention(q.to(DEV), torch.tensor(starts, dtype=torch.int32,
                                                                  device=DEV),
                                         kc, vc, tables.to(DEV), lens.to(DEV), True, SCALE)
        torch.cuda.synchronize()
        for r, (sid, n) in enumerate(chunks):
            ref = _oracle(hist, sid, q[starts[r]:starts[r + 1]], causal=True)
            assert_attention_close(out[starts[r]:starts[r + 1]].cpu().numpy(), ref,
                                   f"prefill of sequence {sid}")

    def decode_step():
        items, pairs = [], []
        for sid in live:
            t = own(1)
            slots, copies = bm.append_tokens(sid, t)
            pairs.extend(copies)
            start = len(hist.chain[sid])
            hist.extend(sid, t)
            items.append((sid, start, start + 1, slots))
        if pairs:
            stats["copies"] += len(pairs)
            pk.copy_blocks(kc, vc, torch.tensor(pairs, dtype=torch.int32, device=DEV))
        _append_rows(pk, hist, items, kc, vc)
        mb = max(len(bm.block_table(s)) for s in live)
        tables, lens = bm.block_tables(live, mb)
        q = rnd(len(live), HQ, D)
        out = pk.paged_decode_attention(q.to(DEV), kc, vc, tables.to(DEV), lens.to(DEV), SCALE,
                                        partition_blocks=2)
        torch.cuda.synchronize()
        for r, sid in enumerate(live):
            assert_attention_close(out[r:r + 1].cpu().numpy(), _oracle(hist, sid, q[r:r + 1], False),
                                   f"decode of sequence {sid}")

    prefill([(0, base[:40] + own(5)), (1, base[:40] + own(9)), (2, base[:33]), (3, own(20))])
    assert stats["hits"] == 2                         # sequences 1 and 2 reuse the prefix
    for step in range(24):
        if step == 2:                                 # parallel samples of partial sequences
            for parent, child in ((0, 10), (1, 11), (2, 12)):
                bm.fork(parent, child)
                hist.extend(child, [], parent=parent)
                live.append(child)
        if step == 9:
            bm.free_sequence(3)
            live.remove(3)
        if step == 10:
            bm.free_sequence(0)
            live.remove(0)
            prefill([(20, base[:40] + own(3)), (21, base[:56] + own(2))])
        decode_step()
    assert stats["copies"] >= 3                       # each fork's first divergent append
    assert pk.get_device_error(clear=True) == 0
    for sid in list(live):
        bm.free_sequence(sid)
    assert bm.num_free_blocks() == NB
