"""Thin ctypes binding over ``libpagedkv.so`` (argument marshalling only).

Every function here checks tensor dtypes/shapes/devices, takes raw device
pointers and the current CUDA stream from torch, and calls the C entry point
of the same name; all compute runs in the library's CUDA kernels.  Importing
this module loads the library and raises if it is missing: there is no
fallback path.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpagedkv.so")

PKV_OK = 0
BLOCK_SIZE = 16

DEVERR_BITS = {
    0x1: "bad slot",
    0x2: "bad block id",
    0x4: "bad context length",
    0x8: "wait timeout",
    0x10: "bad query range",
    0x20: "tensor memory allocation",
    0x40: "query outside f16 range (fp8 decode)",
}


class PagedKVError(RuntimeError):
    """A library call returned a non-zero pkv_status."""

    def __init__(self, func: str, status: int, text: str):
        super().__init__(f"{func} failed with status {status} ({text})")
        self.status = status


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("kv_heads", ctypes.c_int32), ("d_head", ctypes.c_int32)]


_vp, _i32, _i64, _f32, _sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                              ctypes.c_size_t)

SIGNATURES = {
    "pkv_version": ([], ctypes.c_int),
    "pkv_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "pkv_kv_append": ([_vp, _i64, _vp, _i64, _vp, _i64, _vp, _vp, CacheDesc, _vp], ctypes.c_int),
    "pkv_decode_plan": ([ctypes.c_int] * 6 + [ctypes.POINTER(ctypes.c_int),
                                              ctypes.POINTER(ctypes.c_int),
                                              ctypes.POINTER(_sz)], ctypes.c_int),
    "pkv_decode_workspace_bytes": ([ctypes.c_int] * 5, _sz),
    "pkv_paged_decode_attention": ([_vp, ctypes.c_int, ctypes.c_int, _vp, _vp, CacheDesc, _vp,
                                    ctypes.c_int, _vp, ctypes.c_int, _f32, _vp, _vp, _sz, _vp],
                                   ctypes.c_int),
    "pkv_paged_decode_attention_ex": ([_vp, ctypes.c_int, ctypes.c_int, _vp, _vp, CacheDesc, _vp,
                                       ctypes.c_int, _vp, ctypes.c_int, _f32, _vp, _vp, _sz,
                                       ctypes.c_int, _vp], ctypes.c_int),
    "pkv_get_device_error": ([ctypes.POINTER(ctypes.c_uint), ctypes.c_int], ctypes.c_int),
    "pkv_paged_prefill_attention": ([_vp, _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, _vp, _vp, CacheDesc, _vp, ctypes.c_int, _vp,
                                     ctypes.c_int, _f32, _vp, _vp], ctypes.c_int),
    "pkv_kv_append_fp8": ([_vp, _i64, _vp, _i64, _vp, _i64, _vp, _vp, CacheDesc, _f32, _f32,
                           _vp], ctypes.c_int),
    "pkv_paged_decode_attention_fp8": ([_vp, ctypes.c_int, ctypes.c_int, _vp, _vp, CacheDesc, _vp,
                                        ctypes.c_int, _vp, ctypes.c_int, _f32, _f32, _f32, _vp,
                                        _vp, _sz, ctypes.c_int, _vp], ctypes.c_int),
    "pkv_decode_shared_prefix_workspace_bytes": ([ctypes.c_int] * 6, _sz),
    "pkv_paged_decode_attention_shared_prefix": ([_vp, ctypes.c_int, ctypes.c_int, _vp, _vp,
                                                  CacheDesc, _vp, ctypes.c_int, _vp, ctypes.c_int,
                                                  ctypes.c_int, _f32, _vp, _vp, _sz, _vp],
                                                 ctypes.c_int),
    "pkv_noalloc_scratch_bytes": ([], _sz),
    "pkv_paged_decode_attention_noalloc": ([_vp, ctypes.c_int, ctypes.c_int, _vp, _vp, CacheDesc,
                                            _vp, ctypes.c_int, _vp, ctypes.c_int, _f32, _vp,
                                            ctypes.c_int, _vp], ctypes.c_int),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; run `python -m paged_kv_cache_52_gb300.build`"
                           " (the CUDA library is required, there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (args, res) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


lib = _load()


def status_string(status: int) -> str:
    return lib.pkv_status_string(int(status)).decode()


def _check(func: str, status: int):
    if status != PKV_OK:
        raise PagedKVError(func, status, status_string(status))


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(t.data_ptr() if t is not None else 0)


def _need(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def cache_desc(k_cache: torch.Tensor) -> CacheDesc:
    _need(k_cache.dim() == 4, "cache must be [num_blocks, block_size, kv_heads, d_head]")
    nb, bs, hkv, d = k_cache.shape
    return CacheDesc(nb, bs, hkv, d)


def _check_cache(k_cache, v_cache):
    for c in (k_cache, v_cache):
        _need(c.is_cuda and c.dtype == torch.bfloat16 and c.is_contiguous(),
              "caches must be contiguous bf16 CUDA tensors")
    _need(k_cache.shape == v_cache.shape, "k_cache and v_cache shapes differ")


def kv_append(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
              k_cache: torch.Tensor, v_cache: torch.Tensor) -> None:
    """Scatter ``k, v [T, kv_heads, d]`` into the pools at ``slot_mapping [T]`` (-1 skips)."""
    _check_cache(k_cache, v_cache)
    t = slot_mapping.shape[0]
    for x in (k, v):
        _need(x.is_cuda and x.dtype == torch.bfloat16 and x.dim() == 3,
              "k, v must be [T, kv_heads, d] bf16 CUDA tensors")
        _need(x.shape[0] == t and tuple(x.shape[1:]) == tuple(k_cache.shape[2:]),
              "k, v rows must match the cache rows")
        _need(x.stride(2) == 1 and x.stride(1) == x.shape[2],
              "each token row of k, v must be contiguous")
    _need(slot_mapping.is_cuda and slot_mapping.dtype == torch.int64 and
          slot_mapping.is_contiguous(), "slot_mapping must be contiguous int64 on the GPU")
    st = lib.pkv_kv_append(_ptr(k), k.stride(0), _ptr(v), v.stride(0), _ptr(slot_mapping), t,
                           _ptr(k_cache), _ptr(v_cache), cache_desc(k_cache), _stream(k_cache))
    _check("pkv_kv_append", st)


def _check_fp8_cache(k_cache, v_cache):
    for c in (k_cache, v_cache):
        _need(c.is_cuda and c.dtype == torch.uint8 and c.is_contiguous() and c.dim() == 4,
              "FP8 caches must be contiguous uint8 (e4m3 codes) CUDA tensors "
              "[num_blocks, block_size, kv_heads, d_head]")
    _need(k_cache.shape == v_cache.shape, "k_cache and v_cache shapes differ")


def kv_append_fp8(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                  k_cache: torch.Tensor, v_cache: torch.Tensor, k_scale: float,
                  v_scale: float) -> None:
    """Quantize ``k, v [T, kv_heads, d]`` (bf16) to e4m3 with per-pool scales
    and scatter them into the FP8 pools at ``slot_mapping`` (-1 skips)."""
    _check_fp8_cache(k_cache, v_cache)
    t = slot_mapping.shape[0]
    for x in (k, v):
        _need(x.is_cuda and x.dtype == torch.bfloat16 and x.dim() == 3,
              "k, v must be [T, kv_heads, d] bf16 CUDA tensors")
        _need(x.shape[0] == t and tuple(x.shape[1:]) == tuple(k_cache.shape[2:]),
              "k, v rows must match the cache rows")
        _need(x.stride(2) == 1 and x.stride(1) == x.shape[2],
              "each token row of k, v must be contiguous")
    _need(slot_mapping.is_cuda and slot_mapping.dtype == torch.int64 and
          slot_mapping.is_contiguous(), "slot_mapping must be contiguous int64 on the GPU")
    st = lib.pkv_kv_append_fp8(_ptr(k), k.stride(0), _ptr(v), v.stride(0), _ptr(slot_mapping), t,
                               _ptr(k_cache), _ptr(v_cache), cache_desc(k_cache), float(k_scale),
                               float(v_scale), _stream(k_cache))
    _check("pkv_kv_append_fp8", st)


def paged_decode_attention_fp8(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                               block_tables: torch.Tensor, context_lens: torch.Tensor,
                               scale: float, k_scale: float, v_scale: float,
                               out: Optional[torch.Tensor] = None,
                               max_context_len: Optional[int] = None,
                               workspace: Optional[torch.Tensor] = None,
                               partition_blocks: int = 0) -> torch.Tensor:
    """Decode attention over FP8 pools (the dequantized cache's attention)."""
    _check_fp8_cache(k_cache, v_cache)
    _need(q.is_cuda and q.dtype == torch.bfloat16 and q.dim() == 3 and q.is_contiguous(),
          "q must be a contiguous [S, Hq, d] bf16 CUDA tensor")
    S, hq, d = q.shape
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and
          block_tables.is_contiguous() and block_tables.shape[0] == S,
          "block_tables must be contiguous int32 [S, max_blocks]")
    _need(context_lens.dtype == torch.int32 and context_lens.is_contiguous() and
          context_lens.shape == (S,), "context_lens must be contiguous int32 [S]")
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if S else 0
    if out is None:
        out = torch.empty(S, hq, d, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = decode_workspace(S, hq, k_cache.shape[2], d, max_context_len, q.device,
                                     partition_blocks)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib.pkv_paged_decode_attention_fp8(
        _ptr(q), S, hq, _ptr(k_cache), _ptr(v_cache), cache_desc(k_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), int(max_context_len), float(scale),
        float(k_scale), float(v_scale), _ptr(out), _ptr(workspace), ws_bytes,
        int(partition_blocks), _stream(q))
    _check("pkv_paged_decode_attention_fp8", st)
    return out


def decode_plan(num_seqs: int, q_heads: int, kv_heads: int, d_head: int, max_context_len: int,
                partition_blocks: int = 0):
    """(partition_blocks, num_parts, workspace_bytes) the decode will use."""
    pb, np_, ws = ctypes.c_int(), ctypes.c_int(), ctypes.c_size_t()
    st = lib.pkv_decode_plan(num_seqs, q_heads, kv_heads, d_head, max_context_len,
                             partition_blocks, ctypes.byref(pb), ctypes.byref(np_),
                             ctypes.byref(ws))
    _check("pkv_decode_plan", st)
    return pb.value, np_.value, ws.value


def decode_workspace(num_seqs, q_heads, kv_heads, d_head, max_context_len, device,
                     partition_blocks: int = 0) -> Optional[torch.Tensor]:
    """A workspace tensor large enough for the plan (None when not needed)."""
    _, _, ws = decode_plan(num_seqs, q_heads, kv_heads, d_head, max_context_len,
                           partition_blocks)
    if ws == 0:
        return None
    return torch.empty(ws, dtype=torch.uint8, device=device)


def paged_decode_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                           out: Optional[torch.Tensor] = None,
                           max_context_len: Optional[int] = None,
                           workspace: Optional[torch.Tensor] = None,
                           partition_blocks: int = 0) -> torch.Tensor:
    """Decode attention: ``q [S, Hq, d]`` over each sequence's paged history.

    Returns ``out [S, Hq, d]`` float32.  ``max_context_len`` (host int) plans
    the split; when omitted it is read from ``context_lens`` (a device sync).
    """
    _check_cache(k_cache, v_cache)
    _need(q.is_cuda and q.dtype == torch.bfloat16 and q.dim() == 3 and q.is_contiguous(),
          "q must be a contiguous [S, Hq, d] bf16 CUDA tensor")
    S, hq, d = q.shape
    _need(d == k_cache.shape[3], "q and cache head dims differ")
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and
          block_tables.is_contiguous() and block_tables.shape[0] == S,
          "block_tables must be contiguous int32 [S, max_blocks]")
    _need(context_lens.dtype == torch.int32 and context_lens.is_contiguous() and
          context_lens.shape == (S,), "context_lens must be contiguous int32 [S]")
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if S else 0
    if out is None:
        out = torch.empty(S, hq, d, dtype=torch.float32, device=q.device)
    _need(out.dtype == torch.float32 and out.is_contiguous() and out.shape == (S, hq, d),
          "out must be contiguous float32 [S, Hq, d]")
    hkv = k_cache.shape[2]
    if workspace is None:
        workspace = decode_workspace(S, hq, hkv, d, max_context_len, q.device, partition_blocks)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib.pkv_paged_decode_attention_ex(
        _ptr(q), S, hq, _ptr(k_cache), _ptr(v_cache), cache_desc(k_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), int(max_context_len), float(scale), _ptr(out),
        _ptr(workspace), ws_bytes, int(partition_blocks), _stream(q))
    _check("pkv_paged_decode_attention", st)
    return out


def paged_prefill_attention(q: torch.Tensor, q_start: torch.Tensor, k_cache: torch.Tensor,
                            v_cache: torch.Tensor, block_tables: torch.Tensor,
                            context_lens: torch.Tensor, causal: bool, scale: float,
                            out: Optional[torch.Tensor] = None,
                            max_q_len: Optional[int] = None) -> torch.Tensor:
    """Chunked prefill: rows ``q_start[s]:q_start[s+1]`` of ``q [total, Hq, d]``
    are the last tokens of sequence s (already appended).  Returns ``out``
    float32 ``[total, Hq, d]``.  ``max_q_len`` (host int) sizes the grid; when
    omitted it is read from ``q_start`` (a device sync)."""
    _check_cache(k_cache, v_cache)
    _need(q.is_cuda and q.dtype == torch.bfloat16 and q.dim() == 3 and q.is_contiguous(),
          "q must be a contiguous [total, Hq, d] bf16 CUDA tensor")
    total, hq, d = q.shape
    S = context_lens.shape[0]
    _need(q_start.dtype == torch.int32 and q_start.is_contiguous() and q_start.shape == (S + 1,),
          "q_start must be contiguous int32 [S + 1]")
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and
          block_tables.is_contiguous() and block_tables.shape[0] == S,
          "block_tables must be contiguous int32 [S, max_blocks]")
    _need(context_lens.dtype == torch.int32 and context_lens.is_contiguous(),
          "context_lens must be contiguous int32 [S]")
    if max_q_len is None:
        max_q_len = int((q_start[1:] - q_start[:-1]).max().item()) if S else 0
    if out is None:
        out = torch.empty(total, hq, d, dtype=torch.float32, device=q.device)
    _need(out.dtype == torch.float32 and out.is_contiguous() and out.shape == (total, hq, d),
          "out must be contiguous float32 [total, Hq, d]")
    st = lib.pkv_paged_prefill_attention(
        _ptr(q), _ptr(q_start), S, total, int(max_q_len), hq, _ptr(k_cache), _ptr(v_cache),
        cache_desc(k_cache), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
        int(bool(causal)), float(scale), _ptr(out), _stream(q))
    _check("pkv_paged_prefill_attention", st)
    return out


def paged_decode_attention_noalloc(q: torch.Tensor, k_cache: torch.Tensor,
                                   v_cache: torch.Tensor, block_tables: torch.Tensor,
                                   context_lens: torch.Tensor, scale: float, out: torch.Tensor,
                                   max_context_len: int, partition_blocks: int = 0) -> torch.Tensor:
    """Decode attention that allocates nothing: the split-K scratch is the
    library's fixed array (see ``pkv_paged_decode_attention_noalloc``).  The
    caller passes the output buffer; nothing here allocates either."""
    _check_cache(k_cache, v_cache)
    S, hq, d = q.shape
    _need(q.is_cuda and q.dtype == torch.bfloat16 and q.is_contiguous(), "q: contiguous bf16")
    _need(out.dtype == torch.float32 and out.is_contiguous() and out.shape == (S, hq, d),
          "out must be contiguous float32 [S, Hq, d]")
    _need(block_tables.dtype == torch.int32 and block_tables.is_contiguous(),
          "block_tables: contiguous int32")
    _need(context_lens.dtype == torch.int32 and context_lens.is_contiguous(),
          "context_lens: contiguous int32")
    st = lib.pkv_paged_decode_attention_noalloc(
        _ptr(q), S, hq, _ptr(k_cache), _ptr(v_cache), cache_desc(k_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), int(max_context_len), float(scale), _ptr(out),
        int(partition_blocks), _stream(q))
    _check("pkv_paged_decode_attention_noalloc", st)
    return out


def paged_decode_attention_shared_prefix(q: torch.Tensor, k_cache: torch.Tensor,
                                         v_cache: torch.Tensor, block_tables: torch.Tensor,
                                         context_lens: torch.Tensor, scale: float,
                                         prefix_blocks: int, max_context_len: int,
                                         out: Optional[torch.Tensor] = None,
                                         workspace: Optional[torch.Tensor] = None
                                         ) -> torch.Tensor:
    """Decode for sequences whose first ``prefix_blocks`` pages are shared:
    the prefix is attended once for all sequences (tensor cores), the private
    pages by the split-K decode, and the two merged by log-sum-exp."""
    _check_cache(k_cache, v_cache)
    _need(q.is_cuda and q.dtype == torch.bfloat16 and q.dim() == 3 and q.is_contiguous(),
          "q must be a contiguous [S, Hq, d] bf16 CUDA tensor")
    S, hq, d = q.shape
    _need(block_tables.dtype == torch.int32 and block_tables.is_contiguous() and
          block_tables.shape[0] == S, "block_tables must be contiguous int32 [S, max_blocks]")
    _need(context_lens.dtype == torch.int32 and context_lens.is_contiguous(),
          "context_lens must be contiguous int32 [S]")
    if out is None:
        out = torch.empty(S, hq, d, dtype=torch.float32, device=q.device)
    hkv = k_cache.shape[2]
    need = lib.pkv_decode_shared_prefix_workspace_bytes(S, hq, hkv, d, int(max_context_len),
                                                        int(prefix_blocks))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = lib.pkv_paged_decode_attention_shared_prefix(
        _ptr(q), S, hq, _ptr(k_cache), _ptr(v_cache), cache_desc(k_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), int(max_context_len), int(prefix_blocks),
        float(scale), _ptr(out), _ptr(workspace), workspace.numel(), _stream(q))
    _check("pkv_paged_decode_attention_shared_prefix", st)
    return out


def get_device_error(clear: bool = True) -> int:
    """OR of the device-side check bits raised since the last clear (syncs)."""
    word = ctypes.c_uint()
    _check("pkv_get_device_error", lib.pkv_get_device_error(ctypes.byref(word), int(clear)))
    return word.value


def describe_device_error(word: int) -> list[str]:
    return [name for bit, name in DEVERR_BITS.items() if word & bit]
