"""Shared-prefix (cascade) decode: the prefix attended once for all
sequences on the tensor cores, the private pages by split-K (or, for 128 or
more (sequence, KV head) pairs, by the flat split beside the prefix pass on
the library's side stream), merged by log-sum-exp -- equal to the plain
paged decode and to the oracle."""

import pytest
import torch

from paged_kv_cache_52_gb300 import workloads as wl
from parity import DecodeStepOracle, assert_attention_close

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_52_gb300 import pagedkv
    pagedkv.get_device_error(clear=True)
    return pagedkv


def _decodes(m):
    P = m.q_prefill.shape[0]
    return wl.DecodeWorkload("shared-prefix decodes", m.q_decode, m.k_cache, m.v_cache,
                             m.k_new[P:], m.v_new[P:], m.slot_mapping[P:], m.decode_tables,
                             m.decode_lens, m.scale, {"lens": m.meta["decode_lens"]})


def _run(pk, w, prefix_blocks):
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    pk.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    mcl = max(w.meta["lens"])
    casc = pk.paged_decode_attention_shared_prefix(w.q, kc, vc, w.block_tables, w.context_lens,
                                                   w.scale, prefix_blocks, mcl)
    plain = pk.paged_decode_attention(w.q, kc, vc, w.block_tables, w.context_lens, w.scale,
                                      max_context_len=mcl)
    torch.cuda.synchronize()
    return casc, plain


@pytest.mark.parametrize("prefix,ndec,cap", [(64, 40, 600), (16, 7, 100), (1024, 30, 3000)])
def test_shared_prefix_matches_oracle_and_plain_decode(pk, prefix, ndec, cap):
    m = wl.make_mixed_workload(num_prefill=0, num_decode=ndec, shared_prefix=prefix,
                               decode_cap=cap)
    w = _decodes(m)
    ref = DecodeStepOracle(w, range(ndec)).output()
    for n in ("q", "k_cache", "v_cache", "k_new", "v_new", "slot_mapping", "block_tables",
              "context_lens"):
        setattr(w, n, getattr(w, n).to(DEV))
    casc, plain = _run(pk, w, prefix // 16)
    assert_attention_close(casc.cpu().numpy(), ref, f"cascade prefix {prefix}")
    assert_attention_close(casc.cpu().numpy(), plain.cpu().numpy(), "cascade vs plain")
    assert pk.get_device_error() == 0


def test_shared_prefix_full_mixed_step_decodes(pk):
    m = wl.make_mixed_workload(device=DEV, gen_device=DEV)
    w = _decodes(m)
    seqs = list(range(w.num_seqs))
    ref = DecodeStepOracle(w, seqs).output()
    casc, plain = _run(pk, w, m.meta["shared_prefix"] // 16)
    assert_attention_close(casc.cpu().numpy(), ref, "cascade full")
    assert_attention_close(casc.cpu().numpy(), plain.cpu().numpy(), "cascade vs plain full")
    assert pk.get_device_error() == 0


def test_context_shorter_than_prefix_is_flagged_and_decoded_whole(pk):
    m = wl.make_mixed_workload(num_prefill=0, num_decode=4, shared_prefix=64, decode_cap=300)
    w = _decodes(m)
    for n in ("q", "k_cache", "v_cache", "block_tables", "context_lens"):
        setattr(w, n, getattr(w, n).to(DEV))
    lens = w.context_lens.clone()
    lens[2] = 30                      # inside the 64-token prefix
    pk.get_device_error(clear=True)
    out = pk.paged_decode_attention_shared_prefix(w.q, w.k_cache, w.v_cache, w.block_tables,
                                                  lens, w.scale, 4, int(lens.max()))
    plain = pk.paged_decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables, lens, w.scale,
                                      max_context_len=int(lens.max()))
    torch.cuda.synchronize()
    assert pk.get_device_error(clear=True) == PREFIX_MISMATCH
    assert_attention_close(out.cpu().numpy(), plain.cpu().numpy(), "short member, whole context")


# ---- prefix groups: several groups of sequences, each sharing its own prefix
PREFIX_MISMATCH = 0x100


def _grouped_workload(sizes, prefixes, lead_free=1, tail_free=2, hq=16, hkv=4, d=128, seed=31):
    """A decode step over groups of sequences: group g has sizes[g] members
    whose first prefixes[g] pages are the same physical blocks; `lead_free`
    sequences before the groups and `tail_free` after them share nothing.
    Returns (DecodeWorkload on the CPU, group_start, group_prefix_blocks)."""
    g = torch.Generator().manual_seed(seed)
    lens, table_rows, group_start = [], [], [lead_free]
    nb_needed = 0
    plan = [(0, 0)] * lead_free
    for gi, (n, pb) in enumerate(zip(sizes, prefixes)):
        plan += [(gi + 1, pb)] * n
        group_start.append(group_start[-1] + n)
    plan += [(0, 0)] * tail_free
    for grp, pb in plan:
        lens.append(16 * pb + int(torch.randint(1, 300, (1,), generator=g)))
    need = sum(wl.blocks_for(L) for L in lens)
    nb = int(need * 1.25) + 8
    perm = torch.randperm(nb, generator=g).tolist()
    cursor = 0
    shared = {}
    mb = max(wl.blocks_for(L) for L in lens)
    tables = torch.full((len(lens), mb), -1, dtype=torch.int32)
    for s, ((grp, pb), L) in enumerate(zip(plan, lens)):
        if grp and grp not in shared:
            shared[grp] = perm[cursor:cursor + pb]
            cursor += pb
        ids = list(shared[grp]) if grp else []
        own = wl.blocks_for(L) - len(ids)
        ids += perm[cursor:cursor + own]
        cursor += own
        tables[s, :len(ids)] = torch.tensor(ids, dtype=torch.int32)
    S = len(lens)
    kc = (torch.randn(nb, 16, hkv, d, generator=g)).to(torch.bfloat16)
    vc = (torch.randn(nb, 16, hkv, d, generator=g)).to(torch.bfloat16)
    q = torch.randn(S, hq, d, generator=g).to(torch.bfloat16)
    kn = torch.randn(S, hkv, d, generator=g).to(torch.bfloat16)
    vn = torch.randn(S, hkv, d, generator=g).to(torch.bfloat16)
    slots = wl.append_slots(tables, [[L - 1] for L in lens])
    w = wl.DecodeWorkload("prefix groups", q, kc, vc, kn, vn, slots, tables,
                          torch.tensor(lens, dtype=torch.int32), 1.0 / d ** 0.5, {"lens": lens})
    return (w, torch.tensor(group_start, dtype=torch.int32),
            torch.tensor(prefixes, dtype=torch.int32))


def _to_dev(w):
    for n in ("q", "k_cache", "v_cache", "k_new", "v_new", "slot_mapping", "block_tables",
              "context_lens"):
        setattr(w, n, getattr(w, n).to(DEV))
    return w


def _run_groups(pk, w, gs, gp):
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    pk.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    sizes = (gs[1:] - gs[:-1]).tolist()
    out = pk.paged_decode_attention_prefix_groups(
        w.q, kc, vc, w.block_tables, w.context_lens, w.scale, gs.to(DEV), gp.to(DEV),
        max(sizes), int(gp.max()), max(w.meta["lens"]))
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("hq,hkv,d", [(16, 4, 128), (64, 8, 128), (8, 8, 64)])
def test_prefix_groups_match_oracle(pk, hq, hkv, d):
    # four groups (one of a single member), one sequence before them and two after
    w, gs, gp = _grouped_workload([5, 1, 7, 3], [4, 2, 8, 1], hq=hq, hkv=hkv, d=d)
    ref = DecodeStepOracle(w, range(w.num_seqs)).output()
    out = _run_groups(pk, _to_dev(w), gs, gp)
    assert_attention_close(out.cpu().numpy(), ref, f"prefix groups {hq}/{hkv} d{d}")
    assert pk.get_device_error(clear=True) == 0


def test_prefix_group_mismatch_is_flagged_and_decoded_whole(pk):
    w, gs, gp = _grouped_workload([5, 4, 6], [4, 3, 8], lead_free=0, tail_free=1)
    # member 2 of group 0 keeps a private copy of its third prefix page: its
    # ids differ from the leader's, so it is not shared (the content is not
    # the same either, so only decoding its own pages gives the oracle's result)
    used = set(w.block_tables.flatten().tolist())
    spare = next(b for b in range(w.k_cache.shape[0]) if b not in used)
    w.block_tables[2, 2] = spare
    ref = DecodeStepOracle(w, range(w.num_seqs)).output()
    pk.get_device_error(clear=True)
    out = _run_groups(pk, _to_dev(w), gs, gp)
    assert pk.get_device_error(clear=True) == PREFIX_MISMATCH
    assert_attention_close(out.cpu().numpy(), ref, "mismatched member")


def test_prefix_groups_full_mixed_step_whole_batch(pk):
    # the mixed step's 248 decodes as one group sharing the 1024-token prefix,
    # every sequence compared with the oracle
    m = wl.make_mixed_workload(device=DEV, gen_device=DEV)
    w = _decodes(m)
    ref = DecodeStepOracle(w, range(w.num_seqs)).output()
    gs = torch.tensor([0, w.num_seqs], dtype=torch.int32)
    gp = torch.tensor([m.meta["shared_prefix"] // 16], dtype=torch.int32)
    out = _run_groups(pk, w, gs, gp)
    assert_attention_close(out.cpu().numpy(), ref, "prefix group, mixed-step decodes")
    assert pk.get_device_error(clear=True) == 0


# ---- the same with the flat split for the private pages (128 or more
# (sequence, KV head) pairs at d_head 128), the prefix pass beside it


def _assert_flat(pk, w):
    S, hq, d = w.q.shape
    assert pk.decode_plan_uses_flat(S, hq, w.k_cache.shape[2], d, max(w.meta["lens"]), 0)


def test_prefix_groups_flat_suffix_match_oracle(pk):
    w, gs, gp = _grouped_workload([12, 1, 9, 6], [4, 2, 8, 1], hq=64, hkv=8)
    _assert_flat(pk, w)
    ref = DecodeStepOracle(w, range(w.num_seqs)).output()
    out = _run_groups(pk, _to_dev(w), gs, gp)
    assert_attention_close(out.cpu().numpy(), ref, "prefix groups, flat suffix")
    assert pk.get_device_error(clear=True) == 0


def test_prefix_group_mismatch_flat_suffix(pk):
    w, gs, gp = _grouped_workload([8, 6, 10], [4, 3, 8], lead_free=0, tail_free=1, hq=64, hkv=8)
    _assert_flat(pk, w)
    used = set(w.block_tables.flatten().tolist())
    spare = next(b for b in range(w.k_cache.shape[0]) if b not in used)
    w.block_tables[2, 2] = spare                       # a private copy of a prefix page
    ref = DecodeStepOracle(w, range(w.num_seqs)).output()
    pk.get_device_error(clear=True)
    out = _run_groups(pk, _to_dev(w), gs, gp)
    assert pk.get_device_error(clear=True) == PREFIX_MISMATCH
    assert_attention_close(out.cpu().numpy(), ref, "mismatched member, flat suffix")


@pytest.mark.parametrize("prefix", [64, 1024])
def test_shared_prefix_flat_suffix_matches_oracle(pk, prefix):
    # 28 decodes of 64 / 8 heads, some ending right after the prefix
    m = wl.make_mixed_workload(num_prefill=0, num_decode=28, shared_prefix=prefix,
                               decode_cap=prefix + 400)
    w = _decodes(m)
    _assert_flat(pk, w)
    ref = DecodeStepOracle(w, range(w.num_seqs)).output()
    casc, plain = _run(pk, _to_dev(w), prefix // 16)
    assert_attention_close(casc.cpu().numpy(), ref, f"cascade, flat suffix, prefix {prefix}")
    assert_attention_close(casc.cpu().numpy(), plain.cpu().numpy(), "cascade vs plain, flat")
    assert pk.get_device_error() == 0


def test_short_member_flat_suffix(pk):
    m = wl.make_mixed_workload(num_prefill=0, num_decode=28, shared_prefix=64, decode_cap=300)
    w = _to_dev(_decodes(m))
    _assert_flat(pk, w)
    lens = w.context_lens.clone()
    lens[2] = 30                      # inside the 64-token prefix
    lens[5] = 64                      # exactly the prefix: no own page
    pk.get_device_error(clear=True)
    out = pk.paged_decode_attention_shared_prefix(w.q, w.k_cache, w.v_cache, w.block_tables,
                                                  lens, w.scale, 4, int(lens.max()))
    plain = pk.paged_decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables, lens, w.scale,
                                      max_context_len=int(lens.max()))
    torch.cuda.synchronize()
    assert pk.get_device_error(clear=True) == PREFIX_MISMATCH
    assert_attention_close(out.cpu().numpy(), plain.cpu().numpy(), "short members, flat suffix")
