"""The C-ABI library loads, exports every entry point its header declares, and
rejects bad arguments on the host before any launch (no GPU needed)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_52_gb300 import build as b
    if not os.path.exists(b.LIB_PATH):
        b.build()
    from paged_kv_cache_52_gb300 import pagedkv
    return pagedkv


def declared_symbols():
    names = []
    for h in HEADERS:
        text = open(h).read()
        names += re.findall(r"PKV_API\s+[\w\s\*]+?\b(pkv_\w+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_entry_points():
    names = declared_symbols()
    for required in ("pkv_kv_append", "pkv_paged_decode_attention", "pkv_decode_plan",
                     "pkv_get_device_error"):
        assert required in names


def test_library_exports_every_declared_symbol(pk):
    lib = ctypes.CDLL(pk.LIB_PATH)
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing
    # every declared symbol also has a ctypes signature in the binding
    assert set(declared_symbols()) <= set(pk.SIGNATURES), set(declared_symbols()) - set(pk.SIGNATURES)


def test_version_and_status_strings(pk):
    assert pk.lib.pkv_version() >= 100
    assert pk.status_string(0) == "PKV_OK"
    assert "invalid" in pk.status_string(-1)
    assert "unsupported" in pk.status_string(-2)


def _desc(pk, nb=64, bs=16, hkv=2, d=64):
    return pk.CacheDesc(nb, bs, hkv, d)


def test_append_host_validation(pk):
    lib, null = pk.lib, ctypes.c_void_p(0)
    dummy = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first
    assert lib.pkv_kv_append(null, 128, null, 128, null, 0, null, null, _desc(pk), null) == 0
    assert lib.pkv_kv_append(null, 128, null, 128, null, -1, null, null, _desc(pk), null) == -1
    assert lib.pkv_kv_append(dummy, 128, dummy, 128, dummy, 4, null, dummy, _desc(pk), null) == -1
    assert lib.pkv_kv_append(dummy, 128, dummy, 128, dummy, 4, dummy, dummy,
                             _desc(pk, bs=8), null) == -2
    assert lib.pkv_kv_append(dummy, 127, dummy, 128, dummy, 4, dummy, dummy, _desc(pk),
                             null) == -1               # stride below the row / not 16-byte
    assert lib.pkv_kv_append(ctypes.c_void_p((1 << 20) + 2), 128, dummy, 128, dummy, 4, dummy,
                             dummy, _desc(pk), null) == -1  # misaligned base
    assert lib.pkv_kv_append(dummy, 128, dummy, 128, dummy, 4, dummy, dummy,
                             _desc(pk, nb=0), null) == -1


def test_decode_plan_and_workspace(pk):
    pb, parts, ws = pk.decode_plan(4, 8, 2, 64, 1000, partition_blocks=16)
    assert (pb, parts) == (16, 4)                      # ceil(ceil(1000/16) / 16)
    rows = 4 * 8 * parts
    assert ws == (rows * 64 * 4 + 255) // 256 * 256 + rows * 4
    pb, parts, ws = pk.decode_plan(4, 8, 2, 64, 250, partition_blocks=16)
    assert (parts, ws) == (1, 0)
    with pytest.raises(pk.PagedKVError):
        pk.decode_plan(4, 12, 4, 64, 100)              # group 3
    with pytest.raises(pk.PagedKVError):
        pk.decode_plan(4, 8, 2, 96, 100)               # d_head 96
    with pytest.raises(pk.PagedKVError):
        pk.decode_plan(4, 8, 2, 64, 100, partition_blocks=2048)
    with pytest.raises(pk.PagedKVError):
        pk.decode_plan(4, 8, 2, 64, -1)
    # automatic plan, more (sequence, KV head) pairs than CTA slots: partitions
    # of about 150 sqrt(pairs / slots) pages (about 390 for 2048 pairs on 148
    # to 152 SMs), at most what two work items per SM would give
    pb, parts, _ = pk.decode_plan(256, 64, 8, 128, 8192)
    assert 360 <= pb <= 420 and parts == -(-512 // pb)
    pb, _, _ = pk.decode_plan(64, 64, 8, 128, 8192)           # 512 pairs
    assert 180 <= pb <= 210
    pb_small, _, _ = pk.decode_plan(4, 64, 8, 128, 2048)     # few items: short partitions
    assert pb_small == 16
    # few (sequence, KV head) pairs with long contexts: equal partitions that
    # all fit in one wave of two CTAs per SM (at most 1024 pages each)
    pb, parts, _ = pk.decode_plan(4, 64, 8, 128, 131072)
    assert 256 < pb <= 1024 and parts == -(-8192 // pb)
    assert 4 * 8 * parts <= 2 * 152
    assert pk.lib.pkv_decode_workspace_bytes(4, 64, 8, 128, 131072) == \
        pk.decode_plan(4, 64, 8, 128, 131072)[2]


def test_decode_host_validation(pk):
    lib, null = pk.lib, ctypes.c_void_p(0)
    dummy = ctypes.c_void_p(1 << 20)
    args = lambda S, hq, desc, ws=null, wsb=0, pb=16, out=dummy: (  # noqa: E731
        dummy, S, hq, dummy, dummy, desc, dummy, 16, dummy, 250, 0.125, out, ws, wsb, pb, null)
    assert lib.pkv_paged_decode_attention_ex(*args(0, 8, _desc(pk))) == 0      # nothing to do
    assert lib.pkv_paged_decode_attention_ex(*args(4, 8, _desc(pk), out=null)) == -1
    assert lib.pkv_paged_decode_attention_ex(*args(4, 6, _desc(pk))) == -2     # group 3
    assert lib.pkv_paged_decode_attention_ex(*args(4, 8, _desc(pk, bs=32))) == -2
    # split plan (pb=4 -> 4 parts) without a workspace
    assert lib.pkv_paged_decode_attention_ex(*args(4, 8, _desc(pk), pb=4)) == -4


def test_fp8_and_shared_prefix_host_validation(pk):
    lib, null = pk.lib, ctypes.c_void_p(0)
    dummy = ctypes.c_void_p(1 << 20)
    d64 = _desc(pk)                                       # d_head 64: FP8 decode needs 128
    assert lib.pkv_paged_decode_attention_fp8(dummy, 4, 8, dummy, dummy, d64, dummy, 16, dummy,
                                              250, 0.125, 1.0, 1.0, dummy, null, 0, 0,
                                              null) == -2
    # non-positive scales are rejected by the quantizing append
    assert lib.pkv_kv_append_fp8(dummy, 128, dummy, 128, dummy, 4, dummy, dummy, d64, 0.0, 1.0,
                                 null) == -1
    assert lib.pkv_kv_append_fp8(dummy, 128, dummy, 128, dummy, 4, dummy, dummy,
                                 _desc(pk, d=4), 1.0, 1.0, null) == -2   # rows of 16 codes needed
    # a shared prefix of zero pages is not a shared prefix
    assert lib.pkv_decode_shared_prefix_workspace_bytes(4, 8, 2, 64, 250, 0) == 0
    assert lib.pkv_paged_decode_attention_shared_prefix(dummy, 4, 8, dummy, dummy, d64, dummy,
                                                        16, dummy, 250, 0, 0.125, dummy, dummy,
                                                        1 << 20, null) == -1
    # the prefix must fit the block table
    assert lib.pkv_paged_decode_attention_shared_prefix(dummy, 4, 8, dummy, dummy, d64, dummy,
                                                        2, dummy, 250, 4, 0.125, dummy, dummy,
                                                        1 << 30, null) == -1


def test_fp8_prefill_host_validation(pk):
    lib, null = pk.lib, ctypes.c_void_p(0)
    dummy = ctypes.c_void_p(1 << 20)
    d128 = _desc(pk, nb=64, bs=16, hkv=2, d=128)
    need = lib.pkv_paged_prefill_attention_fp8_workspace_bytes(4, 8, 2, 128)
    pool = 4 * 8 * 16 * 2 * 128 * 2                     # bf16 pages of 4 x 8 blocks
    # K, V scratch pools + the table + the persistent launch's work counter
    # + the sequences' dispatch order (4 int32, rounded up to 256 bytes)
    assert need == 2 * pool + 256 + 256 + 256
    assert lib.pkv_paged_prefill_attention_fp8_workspace_bytes(100, 8, 2, 128) == \
        2 * 25 * pool + 3328 + 256 + 512   # table of 800 int32 and order of 100, 256-aligned
    assert lib.pkv_paged_prefill_attention_fp8_workspace_bytes(0, 8, 2, 128) == 0

    def call(desc=d128, k_scale=1.0, v_scale=1.0, ws=dummy, wsb=need, S=4):
        return lib.pkv_paged_prefill_attention_fp8(dummy, dummy, S, 40, 16, 8, dummy, dummy, desc,
                                                   dummy, 8, dummy, 1, 0.1, k_scale, v_scale,
                                                   dummy, ws, wsb, null)
    assert call(S=0) == 0                                 # nothing to do
    assert call(k_scale=0.0) == -1 and call(v_scale=float("inf")) == -1
    assert call(desc=_desc(pk, d=96)) == -2
    assert call(wsb=need - 1) == -4 and call(ws=null) == -4
    assert call(ws=ctypes.c_void_p((1 << 20) + 16)) == -1   # workspace not 256-byte aligned

    def limited(ctas=8, ws=dummy, wsb=need, S=4):
        return lib.pkv_paged_prefill_attention_fp8_limited(dummy, dummy, S, 40, 16, 8, dummy,
                                                           dummy, d128, dummy, 8, dummy, 1, 0.1,
                                                           1.0, 1.0, dummy, ctas, ws, wsb, null)
    assert limited(ctas=0) == -1
    assert limited(ws=null) == -4 and limited(wsb=need - 1) == -4
    assert limited(S=0) == 0


def test_prefill_workspace_host_validation(pk):
    lib, null = pk.lib, ctypes.c_void_p(0)
    dummy = ctypes.c_void_p(1 << 20)
    need = lib.pkv_paged_prefill_workspace_bytes(4, 8, 2, 128)
    # f16 V pages of 4 x 8 blocks + table + the persistent launch's work counter
    # + the dispatch order
    assert need == 4 * 8 * 16 * 2 * 128 * 2 + 256 + 256 + 256
    assert lib.pkv_paged_prefill_workspace_bytes(4, 0, 2, 128) == 0
    d128 = _desc(pk, nb=64, bs=16, hkv=2, d=128)

    def call(ws=dummy, wsb=need, desc=d128):
        return lib.pkv_paged_prefill_attention_ex(dummy, dummy, 4, 40, 16, 8, dummy, dummy, desc,
                                                  dummy, 8, dummy, 1, 0.1, dummy, ws, wsb, null)
    assert call(wsb=need - 1) == -4
    assert call(ws=ctypes.c_void_p((1 << 20) + 64)) == -1  # not 256-byte aligned
    assert call(desc=_desc(pk, d=96)) == -2

    def limited(ctas=8, ws=dummy, wsb=need, desc=d128, S=4):
        return lib.pkv_paged_prefill_attention_limited(dummy, dummy, S, 40, 16, 8, dummy, dummy,
                                                       desc, dummy, 8, dummy, 1, 0.1, dummy, ctas,
                                                       ws, wsb, null)
    assert limited(ctas=0) == -1 and limited(ctas=-3) == -1
    assert limited(ws=null) == -4 and limited(wsb=need - 1) == -4
    assert limited(ws=ctypes.c_void_p((1 << 20) + 64)) == -1
    assert limited(desc=_desc(pk, d=96)) == -2
    assert limited(S=0) == 0                              # nothing to do


def test_bf16_out_host_validation(pk):
    lib, null = pk.lib, ctypes.c_void_p(0)
    dummy = ctypes.c_void_p(1 << 20)
    half_aligned = ctypes.c_void_p((1 << 20) + 2)      # 2-byte aligned, not 4
    dec = lambda fn, S=4, out=dummy, pb=4: fn(  # noqa: E731
        dummy, S, 8, dummy, dummy, _desc(pk), dummy, 16, dummy, 250, 0.125, out, null, 0, pb, null)
    bf = lib.pkv_paged_decode_attention_bf16out
    assert dec(bf, S=0) == 0                                # nothing to do
    assert dec(bf, out=null) == -1
    assert dec(bf, out=ctypes.c_void_p((1 << 20) + 1)) == -1  # a bf16 output needs 2 bytes
    # 2-byte alignment passes for bf16 (the split plan then wants a workspace),
    # while the float32 entry point rejects the same pointer
    assert dec(bf, out=half_aligned) == -4
    assert dec(lib.pkv_paged_decode_attention_ex, out=half_aligned) == -1

    d128 = _desc(pk, nb=64, bs=16, hkv=2, d=128)
    need = lib.pkv_paged_prefill_workspace_bytes(4, 8, 2, 128)

    def pre(ws=dummy, wsb=need, desc=d128, out=dummy, S=4):
        return lib.pkv_paged_prefill_attention_bf16out(dummy, dummy, S, 40, 16, 8, dummy, dummy,
                                                       desc, dummy, 8, dummy, 1, 0.1, out, ws,
                                                       wsb, null)
    assert pre(S=0) == 0 and pre(ws=null, S=0) == 0
    assert pre(out=ctypes.c_void_p((1 << 20) + 8)) == -1   # rows are stored 16 bytes at a time
    assert pre(out=ctypes.c_void_p((1 << 20) + 8), ws=null) == -1
    assert pre(wsb=need - 1) == -4
    assert pre(desc=_desc(pk, d=96)) == -2 and pre(desc=_desc(pk, d=96), ws=null) == -2


def test_checked_append_host_validation(pk):
    lib, null = pk.lib, ctypes.c_void_p(0)
    dummy = ctypes.c_void_p(1 << 20)
    d = _desc(pk, nb=64, bs=16, hkv=2, d=64)             # 1024 slots
    need = lib.pkv_kv_append_checked_workspace_bytes(d)
    assert need == 256 + 256                              # flag, then 32 words of bitmap
    assert lib.pkv_kv_append_checked_workspace_bytes(_desc(pk, nb=1000, bs=16, hkv=2, d=64)) == \
        256 + 2048                                        # 16,000 slots: 500 words, 256-aligned
    assert lib.pkv_kv_append_checked_workspace_bytes(_desc(pk, bs=32)) == 0

    def call(ws=dummy, wsb=need, T=4):
        return lib.pkv_kv_append_checked(dummy, 128, dummy, 128, dummy, T, dummy, dummy, d, ws,
                                         wsb, null)
    assert call(T=0) == 0                                 # nothing to do
    assert call(T=-1) == -1
    assert call(ws=null) == -4 and call(wsb=need - 1) == -4
    assert call(ws=ctypes.c_void_p((1 << 20) + 16)) == -1  # workspace not 256-byte aligned


def test_fp8_decode_and_verify_bf16_out_host_validation(pk):
    lib, null = pk.lib, ctypes.c_void_p(0)
    dummy = ctypes.c_void_p(1 << 20)
    half = ctypes.c_void_p((1 << 20) + 2)                 # 2-byte aligned only
    d128 = _desc(pk, nb=64, bs=16, hkv=2, d=128)
    fp8 = lambda fn, out: fn(dummy, 4, 8, dummy, dummy, d128, dummy, 16, dummy, 250,  # noqa: E731
                             0.125, 1.0, 1.0, out, null, 0, 4, null)
    # 2-byte alignment passes for bf16 (then the split plan wants a workspace)
    assert fp8(lib.pkv_paged_decode_attention_fp8_bf16out, half) == -4
    assert fp8(lib.pkv_paged_decode_attention_fp8, half) == -1
    assert fp8(lib.pkv_paged_decode_attention_fp8_bf16out, ctypes.c_void_p((1 << 20) + 1)) == -1
    ver = lambda fn, out, S=4: fn(dummy, S, 2, 8, dummy, dummy, d128, dummy, 16, dummy,  # noqa: E731
                                  250, 0.125, out, null, 0, 4, null)
    assert ver(lib.pkv_paged_verify_attention_bf16out, half) == -4
    assert ver(lib.pkv_paged_verify_attention, half) == -1
    assert ver(lib.pkv_paged_verify_attention_bf16out, null) == -1
    assert ver(lib.pkv_paged_verify_attention_bf16out, half, S=0) == 0


def test_wait_probe_host_validation(pk):
    lib, null = pk.lib, ctypes.c_void_p(0)
    limit = lib.pkv_wait_poll_limit()
    assert limit == 1 << 18
    assert lib.pkv_wait_timeout_probe(0, null, null) == -1
    assert lib.pkv_wait_timeout_probe(limit + 1, null, null) == -1   # never longer than a real wait
    assert lib.pkv_wait_timeout_probe(16, ctypes.c_void_p((1 << 20) + 4), null) == -1


def test_decode_plan_flat_choice_and_workspace(pk):
    # the library's split over bf16 pages: flat for 193-1024 (sequence, KV
    # head) pairs at d_head 128 and for more pairs in 3 or more uniform
    # partitions; its workspace also covers the uniform split of the same
    # sizes (which the FP8 and verification decodes take) and, from 128
    # pairs, the flat split (which the FP8 decode takes from there)
    assert not pk.decode_plan_uses_flat(8, 64, 8, 128, 8192)
    assert not pk.decode_plan_uses_flat(16, 64, 8, 128, 8192)
    assert pk.decode_plan_uses_flat(32, 64, 8, 128, 8192)
    assert not pk.decode_plan_uses_flat(256, 64, 8, 128, 8192)     # 2 partitions
    assert pk.decode_plan_uses_flat(248, 64, 8, 128, 32768)        # 6 partitions
    assert not pk.decode_plan_uses_flat(32, 64, 8, 64, 8192)       # d_head 64
    for args in ((16, 64, 8, 128, 8192), (32, 64, 8, 128, 8192), (248, 64, 8, 128, 32768),
                 (700, 16, 4, 128, 80)):
        uni = pk.decode_plan(*args, partition_blocks=pk.SPLIT_UNIFORM)[2]
        flat = pk.decode_plan(*args, partition_blocks=pk.SPLIT_FLAT)[2]
        auto = pk.decode_plan(*args)[2]
        assert flat >= uni and auto >= uni
        assert pk.lib.pkv_decode_workspace_bytes(*args) == auto
    assert pk.lib.pkv_decode_plan_uses_flat(2000, 8, 8, 128, 256, pk.SPLIT_FLAT) < 0
