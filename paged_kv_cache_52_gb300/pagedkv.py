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
# partition_blocks values that name a split rule rather than a size
SPLIT_BALANCED = -1   # length-balanced work list (bf16 decode)
SPLIT_UNIFORM = -2    # uniform partitions sized by the library
SPLIT_FLAT = -3       # flat split: each warp streams one contiguous page range (bf16 decode)

DEVERR_BITS = {
    0x1: "bad slot",
    0x2: "bad block id",
    0x4: "bad context length",
    0x8: "wait timeout",
    0x10: "bad query range",
    0x20: "tensor memory allocation",
    0x40: "query outside f16 range (fp8 decode)",
    0x80: "duplicate slot (checked append wrote nothing)",
    0x100: "prefix-group member without its group's prefix (decoded without it)",
}


class PagedKVError(RuntimeError):
    """A library call returned a non-zero pkv_status."""

    def __init__(self, func: str, status: int, text: str):
        super().__init__(f"{func} failed with status {status} ({text})")
        self.status = status


class NoFreeBlocks(PagedKVError):
    """The block pool has fewer free blocks than the operation needs; the
    manager is unchanged."""


PKV_ENOBLOCKS = -8


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("kv_heads", ctypes.c_int32), ("d_head", ctypes.c_int32)]


_vp, _i32, _i64, _f32, _sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                              ctypes.c_size_t)

SIGNATURES = {
    "pkv_version": ([], ctypes.c_int),
    "pkv_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "pkv_kv_append": ([_vp, _i64, _vp, _i64, _vp, _i64, _vp, _vp, CacheDesc, _vp], ctypes.c_int),
    "pkv_kv_append_checked_workspace_bytes": ([CacheDesc], _sz),
    "pkv_kv_append_checked": ([_vp, _i64, _vp, _i64, _vp, _i64, _vp, _vp, CacheDesc, _vp, _sz,
                               _vp], ctypes.c_int),
    "pkv_decode_plan": ([ctypes.c_int] * 6 + [ctypes.POINTER(ctypes.c_int),
                                              ctypes.POINTER(ctypes.c_int),
                                              ctypes.POINTER(_sz)], ctypes.c_int),
    "pkv_decode_workspace_bytes": ([ctypes.c_int] * 5, _sz),
    "pkv_decode_plan_uses_list": ([ctypes.c_int] * 6, ctypes.c_int),
    "pkv_decode_plan_uses_flat": ([ctypes.c_int] * 6, ctypes.c_int),
    "pkv_paged_decode_step": ([_vp, ctypes.c_int, ctypes.c_int, _vp, _i64, _vp, _i64, _vp, _vp,
                               _vp, CacheDesc, _vp, ctypes.c_int, _vp, ctypes.c_int, _f32, _vp,
                               _vp, _sz, _vp], ctypes.c_int),
    "pkv_decode_limited_workspace_bytes": ([ctypes.c_int] * 6, _sz),
    "pkv_mixed_step_workspace_bytes": ([ctypes.c_int] * 7, _sz),
    "pkv_mixed_step_attention": ([_vp, _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp,
                                  ctypes.c_int, _vp, ctypes.c_int, _vp, ctypes.c_int, _vp,
                                  ctypes.c_int, _vp, ctypes.c_int, ctypes.c_int, _vp, _vp,
                                  CacheDesc, _f32, _vp, _vp, _vp, _sz, _vp], ctypes.c_int),
    "pkv_mixed_step_groups_workspace_bytes": ([ctypes.c_int] * 8, _sz),
    "pkv_mixed_step_attention_ex": ([_vp, _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp,
                                     ctypes.c_int, _vp, ctypes.c_int, _vp, ctypes.c_int, _vp,
                                     ctypes.c_int, _vp, ctypes.c_int, ctypes.c_int, _vp, _vp,
                                     CacheDesc, _f32, _vp, _vp, _vp, _vp, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int, _vp, _sz, ctypes.c_int, _vp],
                                    ctypes.c_int),
    "pkv_paged_decode_attention_limited": ([_vp, ctypes.c_int, ctypes.c_int, _vp, _vp, CacheDesc,
                                            _vp, ctypes.c_int, _vp, ctypes.c_int, _f32, _vp,
                                            ctypes.c_int, _vp, _sz, _vp], ctypes.c_int),
    "pkv_paged_decode_attention": ([_vp, ctypes.c_int, ctypes.c_int, _vp, _vp, CacheDesc, _vp,
                                    ctypes.c_int, _vp, ctypes.c_int, _f32, _vp, _vp, _sz, _vp],
                                   ctypes.c_int),
    "pkv_paged_decode_attention_ex": ([_vp, ctypes.c_int, ctypes.c_int, _vp, _vp, CacheDesc, _vp,
                                       ctypes.c_int, _vp, ctypes.c_int, _f32, _vp, _vp, _sz,
                                       ctypes.c_int, _vp], ctypes.c_int),
    "pkv_paged_decode_attention_fp8_bf16out": ([_vp, ctypes.c_int, ctypes.c_int, _vp, _vp,
                                                CacheDesc, _vp, ctypes.c_int, _vp, ctypes.c_int,
                                                _f32, _f32, _f32, _vp, _vp, _sz, ctypes.c_int,
                                                _vp], ctypes.c_int),
    "pkv_paged_verify_attention_bf16out": ([_vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp,
                                            _vp, CacheDesc, _vp, ctypes.c_int, _vp, ctypes.c_int,
                                            _f32, _vp, _vp, _sz, ctypes.c_int, _vp],
                                           ctypes.c_int),
    "pkv_paged_decode_attention_bf16out": ([_vp, ctypes.c_int, ctypes.c_int, _vp, _vp, CacheDesc,
                                            _vp, ctypes.c_int, _vp, ctypes.c_int, _f32, _vp, _vp,
                                            _sz, ctypes.c_int, _vp], ctypes.c_int),
    "pkv_paged_prefill_attention_bf16out": ([_vp, _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, _vp, _vp, CacheDesc, _vp,
                                             ctypes.c_int, _vp, ctypes.c_int, _f32, _vp, _vp, _sz,
                                             _vp], ctypes.c_int),
    "pkv_get_device_error": ([ctypes.POINTER(ctypes.c_uint), ctypes.c_int], ctypes.c_int),
    "pkv_get_last_device_error": ([_vp], ctypes.c_int),
    "pkv_get_last_device_error_bits": ([_vp, ctypes.POINTER(ctypes.c_uint)], ctypes.c_int),
    "pkv_wait_poll_limit": ([], ctypes.c_uint32),
    "pkv_wait_timeout_probe": ([ctypes.c_uint32, _vp, _vp], ctypes.c_int),
    "pkv_paged_prefill_attention": ([_vp, _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, _vp, _vp, CacheDesc, _vp, ctypes.c_int, _vp,
                                     ctypes.c_int, _f32, _vp, _vp], ctypes.c_int),
    "pkv_kv_append_fp8": ([_vp, _i64, _vp, _i64, _vp, _i64, _vp, _vp, CacheDesc, _f32, _f32,
                           _vp], ctypes.c_int),
    "pkv_paged_decode_attention_fp8": ([_vp, ctypes.c_int, ctypes.c_int, _vp, _vp, CacheDesc, _vp,
                                        ctypes.c_int, _vp, ctypes.c_int, _f32, _f32, _f32, _vp,
                                        _vp, _sz, ctypes.c_int, _vp], ctypes.c_int),
    "pkv_decode_shared_prefix_workspace_bytes": ([ctypes.c_int] * 6, _sz),
    "pkv_decode_prefix_groups_workspace_bytes": ([ctypes.c_int] * 6, _sz),
    "pkv_paged_decode_attention_prefix_groups": ([_vp, ctypes.c_int, ctypes.c_int, _vp, _vp,
                                                  CacheDesc, _vp, ctypes.c_int, _vp, ctypes.c_int,
                                                  _vp, _vp, ctypes.c_int, ctypes.c_int,
                                                  ctypes.c_int, _f32, _vp, _vp, _sz, _vp],
                                                 ctypes.c_int),
    "pkv_paged_decode_attention_shared_prefix": ([_vp, ctypes.c_int, ctypes.c_int, _vp, _vp,
                                                  CacheDesc, _vp, ctypes.c_int, _vp, ctypes.c_int,
                                                  ctypes.c_int, _f32, _vp, _vp, _sz, _vp],
                                                 ctypes.c_int),
    "pkv_noalloc_scratch_bytes": ([], _sz),
    "pkv_paged_decode_attention_noalloc": ([_vp, ctypes.c_int, ctypes.c_int, _vp, _vp, CacheDesc,
                                            _vp, ctypes.c_int, _vp, ctypes.c_int, _f32, _vp,
                                            ctypes.c_int, _vp], ctypes.c_int),
    "pkv_paged_prefill_attention_fp8_workspace_bytes": ([ctypes.c_int] * 4, _sz),
    "pkv_paged_prefill_workspace_bytes": ([ctypes.c_int] * 4, _sz),
    "pkv_paged_prefill_attention_ex": ([_vp, _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, _vp, _vp, CacheDesc, _vp, ctypes.c_int, _vp,
                                        ctypes.c_int, _f32, _vp, _vp, _sz, _vp], ctypes.c_int),
    "pkv_paged_prefill_attention_fp8_limited": ([_vp, _vp, ctypes.c_int, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_int, _vp, _vp, CacheDesc,
                                                 _vp, ctypes.c_int, _vp, ctypes.c_int, _f32,
                                                 _f32, _f32, _vp, ctypes.c_int, _vp, _sz, _vp],
                                                ctypes.c_int),
    "pkv_paged_prefill_attention_limited": ([_vp, _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, _vp, _vp, CacheDesc, _vp,
                                             ctypes.c_int, _vp, ctypes.c_int, _f32, _vp,
                                             ctypes.c_int, _vp, _sz, _vp], ctypes.c_int),
    "pkv_paged_prefill_attention_fp8": ([_vp, _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, _vp, _vp, CacheDesc, _vp, ctypes.c_int,
                                         _vp, ctypes.c_int, _f32, _f32, _f32, _vp, _vp, _sz, _vp],
                                        ctypes.c_int),
    "pkv_verify_workspace_bytes": ([ctypes.c_int] * 7, _sz),
    "pkv_paged_verify_attention": ([_vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp, _vp,
                                    CacheDesc, _vp, ctypes.c_int, _vp, ctypes.c_int, _f32, _vp,
                                    _vp, _sz, ctypes.c_int, _vp], ctypes.c_int),
    # host block manager (pagedkv_blocks.h); pointers are host memory
    "pkv_bm_create": ([_i32, _i32, ctypes.POINTER(_vp)], ctypes.c_int),
    "pkv_bm_destroy": ([_vp], None),
    "pkv_bm_add_sequence": ([_vp, _i64, _vp, _i32, ctypes.POINTER(_i32)], ctypes.c_int),
    "pkv_bm_append_tokens": ([_vp, _i64, _vp, _i32, _vp, _vp, _i32, ctypes.POINTER(_i32)],
                             ctypes.c_int),
    "pkv_bm_fork": ([_vp, _i64, _i64], ctypes.c_int),
    "pkv_bm_free_sequence": ([_vp, _i64], ctypes.c_int),
    "pkv_bm_slots": ([_vp, _i64, _i32, _i32, _vp], ctypes.c_int),
    "pkv_bm_seq_len": ([_vp, _i64, ctypes.POINTER(_i32)], ctypes.c_int),
    "pkv_bm_block_table": ([_vp, _i64, _vp, _i32, ctypes.POINTER(_i32)], ctypes.c_int),
    "pkv_bm_block_tables": ([_vp, _vp, _i32, _vp, _i32, _vp], ctypes.c_int),
    "pkv_bm_num_free_blocks": ([_vp], _i32),
    "pkv_bm_refcount": ([_vp, _i32], _i32),
    "pkv_bm_free_list": ([_vp, _vp, _i32, ctypes.POINTER(_i32)], ctypes.c_int),
    "pkv_blocks_for_budget": ([_i64, _i64, _i64, _i32, _i32, _i32, _i32, _i32], _i64),
    "pkv_copy_blocks": ([_vp, _vp, CacheDesc, _i32, _vp, _i32, _vp], ctypes.c_int),
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
    if status == PKV_ENOBLOCKS:
        raise NoFreeBlocks(func, status, status_string(status))
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
              k_cache: torch.Tensor, v_cache: torch.Tensor,
              checked_workspace: Optional[torch.Tensor] = None) -> None:
    """Scatter ``k, v [T, kv_heads, d]`` into the pools at ``slot_mapping [T]`` (-1 skips).

    With ``checked_workspace`` (see ``kv_append_checked_workspace``) the call
    is ``pkv_kv_append_checked``: a mapping that names one slot twice writes
    nothing and sets the duplicate-slot bit of the device error word."""
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
    if checked_workspace is not None:
        ws = checked_workspace
        _need(ws.is_cuda and ws.dtype == torch.uint8 and ws.is_contiguous(),
              "checked_workspace must be a contiguous uint8 CUDA tensor")
        st = lib.pkv_kv_append_checked(_ptr(k), k.stride(0), _ptr(v), v.stride(0),
                                       _ptr(slot_mapping), t, _ptr(k_cache), _ptr(v_cache),
                                       cache_desc(k_cache), _ptr(ws), ws.numel(),
                                       _stream(k_cache))
        _check("pkv_kv_append_checked", st)
        return
    st = lib.pkv_kv_append(_ptr(k), k.stride(0), _ptr(v), v.stride(0), _ptr(slot_mapping), t,
                           _ptr(k_cache), _ptr(v_cache), cache_desc(k_cache), _stream(k_cache))
    _check("pkv_kv_append", st)


def kv_append_checked_workspace(k_cache: torch.Tensor) -> torch.Tensor:
    """Workspace of the checked append for this pool: a flag and one bit per slot."""
    n = lib.pkv_kv_append_checked_workspace_bytes(cache_desc(k_cache))
    _need(n > 0, "unsupported cache shape")
    return torch.empty(n, dtype=torch.uint8, device=k_cache.device)


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
                               partition_blocks: int = 0,
                               out_dtype: Optional[torch.dtype] = None) -> torch.Tensor:
    """Decode attention over FP8 pools (the dequantized cache's attention).
    ``out`` is float32 unless ``out_dtype`` (or a given ``out``) is bfloat16."""
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
    odt = _out_dtype(out, out_dtype)
    if out is None:
        out = torch.empty(S, hq, d, dtype=odt, device=q.device)
    _need(out.dtype == odt and out.is_contiguous() and out.shape == (S, hq, d),
          "out must be contiguous float32 or bfloat16 [S, Hq, d]")
    if workspace is None:
        workspace = decode_workspace(S, hq, k_cache.shape[2], d, max_context_len, q.device,
                                     partition_blocks)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    fn = (lib.pkv_paged_decode_attention_fp8_bf16out if odt == torch.bfloat16
          else lib.pkv_paged_decode_attention_fp8)
    st = fn(
        _ptr(q), S, hq, _ptr(k_cache), _ptr(v_cache), cache_desc(k_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), int(max_context_len), float(scale),
        float(k_scale), float(v_scale), _ptr(out), _ptr(workspace), ws_bytes,
        int(partition_blocks), _stream(q))
    _check(fn.__name__, st)
    return out


def _out_dtype(out: Optional[torch.Tensor], out_dtype: Optional[torch.dtype]) -> torch.dtype:
    odt = out_dtype if out_dtype is not None else (out.dtype if out is not None
                                                    else torch.float32)
    _need(odt in (torch.float32, torch.bfloat16), "out_dtype must be float32 or bfloat16")
    return odt


def decode_plan(num_seqs: int, q_heads: int, kv_heads: int, d_head: int, max_context_len: int,
                partition_blocks: int = 0):
    """(partition_blocks, num_parts, workspace_bytes) the decode will use."""
    pb, np_, ws = ctypes.c_int(), ctypes.c_int(), ctypes.c_size_t()
    st = lib.pkv_decode_plan(num_seqs, q_heads, kv_heads, d_head, max_context_len,
                             partition_blocks, ctypes.byref(pb), ctypes.byref(np_),
                             ctypes.byref(ws))
    _check("pkv_decode_plan", st)
    return pb.value, np_.value, ws.value


def decode_plan_uses_list(num_seqs: int, q_heads: int, kv_heads: int, d_head: int,
                          max_context_len: int, partition_blocks: int = 0) -> bool:
    """Whether the bf16 decode takes the length-balanced work list."""
    st = lib.pkv_decode_plan_uses_list(num_seqs, q_heads, kv_heads, d_head, max_context_len,
                                       partition_blocks)
    if st < 0:
        _check("pkv_decode_plan_uses_list", st)
    return st == 1


def decode_plan_uses_flat(num_seqs: int, q_heads: int, kv_heads: int, d_head: int,
                          max_context_len: int, partition_blocks: int = 0) -> bool:
    """Whether the bf16 decode takes the flat split."""
    st = lib.pkv_decode_plan_uses_flat(num_seqs, q_heads, kv_heads, d_head, max_context_len,
                                       partition_blocks)
    if st < 0:
        _check("pkv_decode_plan_uses_flat", st)
    return st == 1


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
                           partition_blocks: int = 0,
                           out_dtype: Optional[torch.dtype] = None) -> torch.Tensor:
    """Decode attention: ``q [S, Hq, d]`` over each sequence's paged history.

    Returns ``out [S, Hq, d]``, float32 unless ``out_dtype`` (or a given
    ``out``) is bfloat16: then the float32 result rounded to bf16 in the
    kernel's store (``pkv_paged_decode_attention_bf16out``).
    ``max_context_len`` (host int) plans the split; when omitted it is read
    from ``context_lens`` (a device sync).
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
    odt = _out_dtype(out, out_dtype)
    if out is None:
        out = torch.empty(S, hq, d, dtype=odt, device=q.device)
    _need(out.dtype == odt and out.is_contiguous() and out.shape == (S, hq, d),
          "out must be contiguous float32 or bfloat16 [S, Hq, d]")
    hkv = k_cache.shape[2]
    if workspace is None:
        workspace = decode_workspace(S, hq, hkv, d, max_context_len, q.device, partition_blocks)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    if odt == torch.bfloat16:
        st = lib.pkv_paged_decode_attention_bf16out(
            _ptr(q), S, hq, _ptr(k_cache), _ptr(v_cache), cache_desc(k_cache),
            _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), int(max_context_len),
            float(scale), _ptr(out), _ptr(workspace), ws_bytes, int(partition_blocks), _stream(q))
        _check("pkv_paged_decode_attention_bf16out", st)
        return out
    st = lib.pkv_paged_decode_attention_ex(
        _ptr(q), S, hq, _ptr(k_cache), _ptr(v_cache), cache_desc(k_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), int(max_context_len), float(scale), _ptr(out),
        _ptr(workspace), ws_bytes, int(partition_blocks), _stream(q))
    _check("pkv_paged_decode_attention", st)
    return out


def paged_decode_step(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                      slot_mapping: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                      out: Optional[torch.Tensor] = None,
                      max_context_len: Optional[int] = None,
                      workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """One decode step (``pkv_paged_decode_step``): append each sequence's new
    token (row s of k_new / v_new at slot_mapping[s]) and attend, the append
    hidden under the attention.  float32 ``out [S, Hq, d]``."""
    _check_cache(k_cache, v_cache)
    _need(q.is_cuda and q.dtype == torch.bfloat16 and q.dim() == 3 and q.is_contiguous(),
          "q must be a contiguous [S, Hq, d] bf16 CUDA tensor")
    S, hq, d = q.shape
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _need(t.dtype == torch.bfloat16 and t.dim() == 3 and t.shape[0] == S and
              t.shape[1:] == k_cache.shape[2:] and t.stride(2) == 1 and t.stride(1) == d,
              f"{n} must be [S, Hkv, d] bf16 with contiguous rows")
    _need(slot_mapping.dtype == torch.int64 and slot_mapping.shape == (S,) and
          slot_mapping.is_contiguous(), "slot_mapping must be contiguous int64 [S]")
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
        workspace = decode_workspace(S, hq, k_cache.shape[2], d, max_context_len, q.device)
    ws_bytes = workspace.numel() if workspace is not None else 0
    st = lib.pkv_paged_decode_step(
        _ptr(q), S, hq, _ptr(k_new), k_new.stride(0), _ptr(v_new), v_new.stride(0),
        _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), cache_desc(k_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), int(max_context_len), float(scale), _ptr(out),
        _ptr(workspace), ws_bytes, _stream(q))
    _check("pkv_paged_decode_step", st)
    return out


def decode_limited_workspace(num_seqs, q_heads, kv_heads, d_head, max_context_len, max_ctas,
                             device) -> torch.Tensor:
    n = lib.pkv_decode_limited_workspace_bytes(int(num_seqs), int(q_heads), int(kv_heads),
                                               int(d_head), int(max_context_len), int(max_ctas))
    _need(n > 0, "unsupported limited-decode shape (more than 512 sequences?)")
    return torch.empty(n, dtype=torch.uint8, device=device)


def paged_decode_attention_limited(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                   block_tables: torch.Tensor, context_lens: torch.Tensor,
                                   scale: float, max_ctas: int,
                                   out: Optional[torch.Tensor] = None,
                                   max_context_len: Optional[int] = None,
                                   workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The bf16 decode on at most ``max_ctas`` CTAs (length-balanced list;
    ``pkv_paged_decode_attention_limited``).  float32 ``out [S, Hq, d]``."""
    _check_cache(k_cache, v_cache)
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
    _need(out.dtype == torch.float32 and out.is_contiguous() and out.shape == (S, hq, d),
          "out must be contiguous float32 [S, Hq, d]")
    if workspace is None:
        workspace = decode_limited_workspace(S, hq, k_cache.shape[2], d, max_context_len,
                                             max_ctas, q.device)
    st = lib.pkv_paged_decode_attention_limited(
        _ptr(q), S, hq, _ptr(k_cache), _ptr(v_cache), cache_desc(k_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), int(max_context_len), float(scale), _ptr(out),
        int(max_ctas), _ptr(workspace), workspace.numel(), _stream(q))
    _check("pkv_paged_decode_attention_limited", st)
    return out


def mixed_step_workspace(num_prefill: int, prefill_max_blocks: int, num_decode: int,
                         q_heads: int, kv_heads: int, d_head: int, max_decode_context_len: int,
                         device, num_groups: int = 0) -> torch.Tensor:
    n = lib.pkv_mixed_step_groups_workspace_bytes(int(num_prefill), int(prefill_max_blocks),
                                                  int(num_decode), int(q_heads), int(kv_heads),
                                                  int(d_head), int(max_decode_context_len),
                                                  int(num_groups))
    _need(n > 0, "unsupported mixed-step shape (more than 512 decode sequences?)")
    return torch.empty(n, dtype=torch.uint8, device=device)


def mixed_step_attention(q_prefill: torch.Tensor, q_start: torch.Tensor,
                         prefill_block_tables: torch.Tensor, prefill_context_lens: torch.Tensor,
                         causal: bool, q_decode: torch.Tensor, decode_block_tables: torch.Tensor,
                         decode_context_lens: torch.Tensor, k_cache: torch.Tensor,
                         v_cache: torch.Tensor, scale: float, max_q_len: int,
                         max_decode_context_len: int,
                         out_prefill: Optional[torch.Tensor] = None,
                         out_decode: Optional[torch.Tensor] = None,
                         workspace: Optional[torch.Tensor] = None,
                         prefill_span_permille: int = 0,
                         decode_groups: Optional[tuple] = None):
    """One continuous-batching step's attention in one persistent launch
    (``pkv_mixed_step_attention_ex``): the chunked prefill and the decodes
    over the same pools.  Returns ``(out_prefill, out_decode)``, float32.
    ``prefill_span_permille``: the work list's interleave (0 = the library's).
    ``decode_groups``: optional ``(group_start, group_prefix_blocks,
    max_group_size, max_prefix_blocks)`` -- decode prefix groups as in
    ``paged_decode_attention_prefix_groups`` (int32 device tensors)."""
    _check_cache(k_cache, v_cache)
    for t, n in ((q_prefill, "q_prefill"), (q_decode, "q_decode")):
        _need(t.is_cuda and t.dtype == torch.bfloat16 and t.dim() == 3 and t.is_contiguous(),
              f"{n} must be a contiguous [rows, Hq, d] bf16 CUDA tensor")
    T, hq, d = q_prefill.shape
    S = q_decode.shape[0]
    P = q_start.shape[0] - 1
    for t, n, rows in ((prefill_block_tables, "prefill_block_tables", P),
                       (decode_block_tables, "decode_block_tables", S)):
        _need(t.dtype == torch.int32 and t.dim() == 2 and t.is_contiguous() and t.shape[0] == rows,
              f"{n} must be contiguous int32 [{rows}, max_blocks]")
    for t, n, rows in ((q_start, "q_start", P + 1), (prefill_context_lens, "prefill_context_lens", P),
                       (decode_context_lens, "decode_context_lens", S)):
        _need(t.dtype == torch.int32 and t.is_contiguous() and t.shape == (rows,),
              f"{n} must be contiguous int32 [{rows}]")
    if out_prefill is None:
        out_prefill = torch.empty(T, hq, d, dtype=torch.float32, device=q_prefill.device)
    if out_decode is None:
        out_decode = torch.empty(S, hq, d, dtype=torch.float32, device=q_prefill.device)
    gs = gp = None
    G = mg = mp = 0
    if decode_groups is not None:
        gs, gp, mg, mp = decode_groups
        G = gs.shape[0] - 1
        for t, n, rows in ((gs, "group_start", G + 1), (gp, "group_prefix_blocks", G)):
            _need(t.dtype == torch.int32 and t.is_contiguous() and t.shape == (rows,),
                  f"{n} must be contiguous int32 [{rows}]")
    if workspace is None:
        workspace = mixed_step_workspace(P, prefill_block_tables.shape[1], S, hq,
                                         k_cache.shape[2], d, max_decode_context_len,
                                         q_prefill.device, G)
    st = lib.pkv_mixed_step_attention_ex(
        _ptr(q_prefill), _ptr(q_start), P, T, int(max_q_len), _ptr(prefill_block_tables),
        prefill_block_tables.shape[1], _ptr(prefill_context_lens), int(bool(causal)),
        _ptr(q_decode), S, _ptr(decode_block_tables), decode_block_tables.shape[1],
        _ptr(decode_context_lens), int(max_decode_context_len), hq, _ptr(k_cache), _ptr(v_cache),
        cache_desc(k_cache), float(scale), _ptr(out_prefill), _ptr(out_decode), _ptr(gs),
        _ptr(gp), G, int(mg), int(mp), _ptr(workspace), workspace.numel(),
        int(prefill_span_permille), _stream(q_prefill))
    _check("pkv_mixed_step_attention_ex", st)
    return out_prefill, out_decode


def prefill_workspace(num_seqs: int, max_blocks_per_seq: int, kv_heads: int, d_head: int,
                      device) -> torch.Tensor:
    """Workspace for ``paged_prefill_attention(..., workspace=...)``: the
    chunks' V pages in f16 and their table."""
    n = lib.pkv_paged_prefill_workspace_bytes(int(num_seqs), int(max_blocks_per_seq),
                                              int(kv_heads), int(d_head))
    _need(n > 0, "unsupported prefill workspace shape")
    return torch.empty(n, dtype=torch.uint8, device=device)


def paged_prefill_attention(q: torch.Tensor, q_start: torch.Tensor, k_cache: torch.Tensor,
                            v_cache: torch.Tensor, block_tables: torch.Tensor,
                            context_lens: torch.Tensor, causal: bool, scale: float,
                            out: Optional[torch.Tensor] = None,
                            max_q_len: Optional[int] = None,
                            workspace: Optional[torch.Tensor] = None,
                            max_ctas: Optional[int] = None,
                            out_dtype: Optional[torch.dtype] = None) -> torch.Tensor:
    """Chunked prefill: rows ``q_start[s]:q_start[s+1]`` of ``q [total, Hq, d]``
    are the last tokens of sequence s (already appended).  Returns ``out``
    ``[total, Hq, d]``, float32 unless ``out_dtype`` (or a given ``out``) is
    bfloat16: then the float32 result rounded to bf16 in the kernel's store
    (``pkv_paged_prefill_attention_bf16out``; not with ``max_ctas``).  ``max_q_len`` (host int) sizes the grid; when
    omitted it is read from ``q_start`` (a device sync).  With a ``workspace``
    (see ``prefill_workspace``) the V pages are converted to f16 first and the
    faster single-product P V kernel runs.  ``max_ctas`` (needs the workspace)
    runs that kernel on at most that many SMs, leaving the rest to work on
    other streams (``pkv_paged_prefill_attention_limited``)."""
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
    odt = _out_dtype(out, out_dtype)
    if out is None:
        out = torch.empty(total, hq, d, dtype=odt, device=q.device)
    _need(out.dtype == odt and out.is_contiguous() and out.shape == (total, hq, d),
          "out must be contiguous float32 or bfloat16 [total, Hq, d]")
    _need(max_ctas is None or workspace is not None, "max_ctas needs a workspace")
    _need(max_ctas is None or odt == torch.float32, "max_ctas writes float32 only")
    if workspace is not None:
        _need(workspace.dtype == torch.uint8 and workspace.is_cuda and workspace.is_contiguous(),
              "workspace must be a contiguous uint8 CUDA tensor")
    if odt == torch.bfloat16:
        st = lib.pkv_paged_prefill_attention_bf16out(
            _ptr(q), _ptr(q_start), S, total, int(max_q_len), hq, _ptr(k_cache), _ptr(v_cache),
            cache_desc(k_cache), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
            int(bool(causal)), float(scale), _ptr(out), _ptr(workspace),
            workspace.numel() if workspace is not None else 0, _stream(q))
        _check("pkv_paged_prefill_attention_bf16out", st)
        return out
    if workspace is None:
        st = lib.pkv_paged_prefill_attention(
            _ptr(q), _ptr(q_start), S, total, int(max_q_len), hq, _ptr(k_cache), _ptr(v_cache),
            cache_desc(k_cache), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
            int(bool(causal)), float(scale), _ptr(out), _stream(q))
        _check("pkv_paged_prefill_attention", st)
        return out
    _need(workspace.dtype == torch.uint8 and workspace.is_cuda and workspace.is_contiguous(),
          "workspace must be a contiguous uint8 CUDA tensor")
    if max_ctas is not None:
        st = lib.pkv_paged_prefill_attention_limited(
            _ptr(q), _ptr(q_start), S, total, int(max_q_len), hq, _ptr(k_cache), _ptr(v_cache),
            cache_desc(k_cache), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
            int(bool(causal)), float(scale), _ptr(out), int(max_ctas), _ptr(workspace),
            workspace.numel(), _stream(q))
        _check("pkv_paged_prefill_attention_limited", st)
        return out
    st = lib.pkv_paged_prefill_attention_ex(
        _ptr(q), _ptr(q_start), S, total, int(max_q_len), hq, _ptr(k_cache), _ptr(v_cache),
        cache_desc(k_cache), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
        int(bool(causal)), float(scale), _ptr(out), _ptr(workspace), workspace.numel(),
        _stream(q))
    _check("pkv_paged_prefill_attention_ex", st)
    return out


def paged_prefill_attention_fp8(q: torch.Tensor, q_start: torch.Tensor, k_cache: torch.Tensor,
                                v_cache: torch.Tensor, block_tables: torch.Tensor,
                                context_lens: torch.Tensor, causal: bool, scale: float,
                                k_scale: float, v_scale: float,
                                out: Optional[torch.Tensor] = None,
                                max_q_len: Optional[int] = None,
                                workspace: Optional[torch.Tensor] = None,
                                max_ctas: Optional[int] = None) -> torch.Tensor:
    """Chunked prefill over FP8 (e4m3) pools with per-pool scales: the
    attention of the dequantized cache.  ``workspace`` (uint8, at least
    ``prefill_fp8_workspace_bytes(...)``) holds the widened pages.
    ``max_ctas`` runs the tensor-core prefill on at most that many SMs
    (``pkv_paged_prefill_attention_fp8_limited``)."""
    _check_fp8_cache(k_cache, v_cache)
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
    need = prefill_fp8_workspace_bytes(S, block_tables.shape[1], k_cache.shape[2], d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if max_ctas is not None:
        st = lib.pkv_paged_prefill_attention_fp8_limited(
            _ptr(q), _ptr(q_start), S, total, int(max_q_len), hq, _ptr(k_cache), _ptr(v_cache),
            cache_desc(k_cache), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
            int(bool(causal)), float(scale), float(k_scale), float(v_scale), _ptr(out),
            int(max_ctas), _ptr(workspace), workspace.numel(), _stream(q))
        _check("pkv_paged_prefill_attention_fp8_limited", st)
        return out
    st = lib.pkv_paged_prefill_attention_fp8(
        _ptr(q), _ptr(q_start), S, total, int(max_q_len), hq, _ptr(k_cache), _ptr(v_cache),
        cache_desc(k_cache), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
        int(bool(causal)), float(scale), float(k_scale), float(v_scale), _ptr(out),
        _ptr(workspace), workspace.numel(), _stream(q))
    _check("pkv_paged_prefill_attention_fp8", st)
    return out


def prefill_fp8_workspace_bytes(num_seqs: int, max_blocks_per_seq: int, kv_heads: int,
                                d_head: int) -> int:
    return lib.pkv_paged_prefill_attention_fp8_workspace_bytes(
        int(num_seqs), int(max_blocks_per_seq), int(kv_heads), int(d_head))


def verify_workspace(num_seqs: int, q_len: int, q_heads: int, kv_heads: int, d_head: int,
                     max_context_len: int, device, partition_blocks: int = 0):
    """Workspace for ``paged_verify_attention`` (None when no split is planned)."""
    n = lib.pkv_verify_workspace_bytes(int(num_seqs), int(q_len), int(q_heads), int(kv_heads),
                                       int(d_head), int(max_context_len), int(partition_blocks))
    return torch.empty(n, dtype=torch.uint8, device=device) if n else None


def paged_verify_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                           out: Optional[torch.Tensor] = None,
                           max_context_len: Optional[int] = None,
                           workspace: Optional[torch.Tensor] = None,
                           partition_blocks: int = 0,
                           out_dtype: Optional[torch.dtype] = None) -> torch.Tensor:
    """Speculative verification: ``q [S, K, Hq, d]`` holds the last K tokens of
    each sequence (already appended); token t attends causally over the first
    ``context_len - K + t + 1`` positions.  Returns ``out [S, K, Hq, d]``,
    float32 unless ``out_dtype`` (or a given ``out``) is bfloat16."""
    _check_cache(k_cache, v_cache)
    _need(q.is_cuda and q.dtype == torch.bfloat16 and q.dim() == 4 and q.is_contiguous(),
          "q must be a contiguous [S, K, Hq, d] bf16 CUDA tensor")
    S, K, hq, d = q.shape
    _need(d == k_cache.shape[3], "q and cache head dims differ")
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and
          block_tables.is_contiguous() and block_tables.shape[0] == S,
          "block_tables must be contiguous int32 [S, max_blocks]")
    _need(context_lens.dtype == torch.int32 and context_lens.is_contiguous() and
          context_lens.shape == (S,), "context_lens must be contiguous int32 [S]")
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if S else 0
    odt = _out_dtype(out, out_dtype)
    if out is None:
        out = torch.empty(S, K, hq, d, dtype=odt, device=q.device)
    _need(out.dtype == odt and out.is_contiguous() and out.shape == (S, K, hq, d),
          "out must be contiguous float32 or bfloat16 [S, K, Hq, d]")
    if workspace is None:
        workspace = verify_workspace(S, K, hq, k_cache.shape[2], d, max_context_len, q.device,
                                     partition_blocks)
    fn = (lib.pkv_paged_verify_attention_bf16out if odt == torch.bfloat16
          else lib.pkv_paged_verify_attention)
    st = fn(
        _ptr(q), S, K, hq, _ptr(k_cache), _ptr(v_cache), cache_desc(k_cache),
        _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), int(max_context_len),
        float(scale), _ptr(out), _ptr(workspace), workspace.numel() if workspace is not None else 0,
        int(partition_blocks), _stream(q))
    _check(fn.__name__, st)
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
    pages by the library's split (uniform or flat), and the two merged by
    log-sum-exp."""
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


def paged_decode_attention_prefix_groups(q: torch.Tensor, k_cache: torch.Tensor,
                                         v_cache: torch.Tensor, block_tables: torch.Tensor,
                                         context_lens: torch.Tensor, scale: float,
                                         group_start: torch.Tensor,
                                         group_prefix_blocks: torch.Tensor, max_group_size: int,
                                         max_prefix_blocks: int, max_context_len: int,
                                         out: Optional[torch.Tensor] = None,
                                         workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Decode with groups of sequences sharing their first pages
    (``pkv_paged_decode_attention_prefix_groups``): group g is sequences
    ``group_start[g] .. group_start[g+1]-1`` sharing ``group_prefix_blocks[g]``
    pages.  float32 ``out [S, Hq, d]``."""
    _check_cache(k_cache, v_cache)
    S, hq, d = q.shape
    G = group_start.shape[0] - 1
    _need(q.is_cuda and q.dtype == torch.bfloat16 and q.is_contiguous(), "q: contiguous bf16")
    for t, n, rows in ((group_start, "group_start", G + 1),
                       (group_prefix_blocks, "group_prefix_blocks", G)):
        _need(t.dtype == torch.int32 and t.is_contiguous() and t.shape == (rows,),
              f"{n} must be contiguous int32 [{rows}]")
    if out is None:
        out = torch.empty(S, hq, d, dtype=torch.float32, device=q.device)
    if workspace is None:
        n = lib.pkv_decode_prefix_groups_workspace_bytes(S, hq, k_cache.shape[2], d,
                                                         int(max_context_len), G)
        _need(n > 0, "unsupported prefix-group shape")
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
    st = lib.pkv_paged_decode_attention_prefix_groups(
        _ptr(q), S, hq, _ptr(k_cache), _ptr(v_cache), cache_desc(k_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), int(max_context_len), _ptr(group_start),
        _ptr(group_prefix_blocks), G, int(max_group_size), int(max_prefix_blocks), float(scale),
        _ptr(out), _ptr(workspace), workspace.numel(), _stream(q))
    _check("pkv_paged_decode_attention_prefix_groups", st)
    return out


def get_device_error(clear: bool = True) -> int:
    """OR of the device-side check bits raised since the last clear (syncs)."""
    word = ctypes.c_uint()
    _check("pkv_get_device_error", lib.pkv_get_device_error(ctypes.byref(word), int(clear)))
    return word.value


PKV_EDEVICE_CHECK = -5
PKV_ETIMEOUT = -6


def get_last_device_error(stream: Optional[torch.cuda.Stream] = None) -> tuple[int, int]:
    """Stream-ordered checked-mode status (``pkv_get_last_device_error_bits``):
    waits for the work queued on ``stream`` (torch's current stream by
    default), takes and clears the device error words, and returns
    ``(status, bits)`` with status PKV_OK, PKV_ETIMEOUT or PKV_EDEVICE_CHECK.
    Raises PagedKVError only when the query itself fails."""
    st_ptr = (stream if stream is not None else torch.cuda.current_stream()).cuda_stream
    word = ctypes.c_uint()
    status = lib.pkv_get_last_device_error_bits(ctypes.c_void_p(st_ptr), ctypes.byref(word))
    if status not in (PKV_OK, PKV_ETIMEOUT, PKV_EDEVICE_CHECK):
        _check("pkv_get_last_device_error_bits", status)
    return status, word.value


def wait_timeout_probe(polls: int, device=None) -> int:
    """Run the library's bounded mbarrier wait on a phase that never
    completes, with ``polls`` as the limit (``pkv_wait_timeout_probe``).
    Returns the clock64 cycles the wait took; the timeout bit is left in the
    device error word for the caller to read."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    cycles = torch.zeros(1, dtype=torch.int64, device=dev)
    st = lib.pkv_wait_timeout_probe(int(polls), _ptr(cycles), _stream(cycles))
    _check("pkv_wait_timeout_probe", st)
    return int(cycles.item())


def describe_device_error(word: int) -> list[str]:
    return [name for bit, name in DEVERR_BITS.items() if word & bit]


# --------------------------------------------------------------------------
# Host block manager (pagedkv_blocks.h) and the copy-on-write block copy.
# --------------------------------------------------------------------------
def _i32_host(values) -> "ctypes.Array":
    vals = list(values)
    return (ctypes.c_int32 * max(1, len(vals)))(*vals)


class BlockManager:
    """Handle on the library's native block manager: a pool of
    ``num_blocks`` blocks of ``block_size`` tokens, sequences with block
    tables, prefix sharing by chained hash, forks and copy-on-write.  All
    bookkeeping runs in the library; this class only marshals arguments."""

    def __init__(self, num_blocks: int, block_size: int = BLOCK_SIZE):
        h = ctypes.c_void_p()
        _check("pkv_bm_create", lib.pkv_bm_create(int(num_blocks), int(block_size),
                                                  ctypes.byref(h)))
        self._h = h
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)

    def close(self):
        if self._h:
            lib.pkv_bm_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add_sequence(self, seq_id: int, token_ids) -> int:
        """Blocks for a new prompt; returns the count of leading prompt tokens
        already held by shared blocks."""
        ids = list(token_ids)
        cached = ctypes.c_int32()
        _check("pkv_bm_add_sequence", lib.pkv_bm_add_sequence(
            self._h, int(seq_id), _i32_host(ids), len(ids), ctypes.byref(cached)))
        return cached.value

    def append_tokens(self, seq_id: int, token_ids):
        """Slots for new tokens, and the (src, dst) block copies to make first."""
        ids = list(token_ids)
        slots = (ctypes.c_int64 * max(1, len(ids)))()
        pairs = (ctypes.c_int32 * 2)()
        n = ctypes.c_int32()
        _check("pkv_bm_append_tokens", lib.pkv_bm_append_tokens(
            self._h, int(seq_id), _i32_host(ids), len(ids), slots, pairs, 1, ctypes.byref(n)))
        return list(slots[:len(ids)]), [(pairs[0], pairs[1])] if n.value else []

    def fork(self, parent: int, child: int) -> None:
        _check("pkv_bm_fork", lib.pkv_bm_fork(self._h, int(parent), int(child)))

    def free_sequence(self, seq_id: int) -> None:
        _check("pkv_bm_free_sequence", lib.pkv_bm_free_sequence(self._h, int(seq_id)))

    def slots(self, seq_id: int, start: int, count: int):
        out = (ctypes.c_int64 * max(1, count))()
        _check("pkv_bm_slots", lib.pkv_bm_slots(self._h, int(seq_id), int(start), int(count), out))
        return list(out[:count])

    def seq_len(self, seq_id: int) -> int:
        n = ctypes.c_int32()
        _check("pkv_bm_seq_len", lib.pkv_bm_seq_len(self._h, int(seq_id), ctypes.byref(n)))
        return n.value

    def block_table(self, seq_id: int):
        n = ctypes.c_int32()
        lib.pkv_bm_block_table(self._h, int(seq_id), None, 0, ctypes.byref(n))
        out = (ctypes.c_int32 * max(1, n.value))()
        _check("pkv_bm_block_table", lib.pkv_bm_block_table(self._h, int(seq_id), out, n.value,
                                                            ctypes.byref(n)))
        return list(out[:n.value])

    def block_tables(self, seq_ids, max_blocks_per_seq: int):
        """``(block_tables [S, max_blocks] int32, context_lens [S] int32)`` as
        CPU tensors, in the layout the attention calls take (pad with 0)."""
        ids = list(seq_ids)
        S = len(ids)
        tables = torch.zeros(S, int(max_blocks_per_seq), dtype=torch.int32)
        lens = torch.zeros(S, dtype=torch.int32)
        id_arr = (ctypes.c_int64 * max(1, S))(*ids)
        _check("pkv_bm_block_tables", lib.pkv_bm_block_tables(
            self._h, id_arr, S, _ptr(tables), int(max_blocks_per_seq), _ptr(lens)))
        return tables, lens

    def num_free_blocks(self) -> int:
        return lib.pkv_bm_num_free_blocks(self._h)

    def refcount(self, block: int) -> int:
        return lib.pkv_bm_refcount(self._h, int(block))

    def free_list(self):
        n = ctypes.c_int32()
        out = (ctypes.c_int32 * max(1, self.num_blocks))()
        _check("pkv_bm_free_list", lib.pkv_bm_free_list(self._h, out, self.num_blocks,
                                                        ctypes.byref(n)))
        return list(out[:n.value])


def blocks_for_budget(usable_bytes: int, model_bytes: int, activation_peak_bytes: int,
                      num_layers: int, block_size: int, kv_heads: int, d_head: int,
                      dtype_size: int) -> int:
    n = lib.pkv_blocks_for_budget(int(usable_bytes), int(model_bytes), int(activation_peak_bytes),
                                  int(num_layers), int(block_size), int(kv_heads), int(d_head),
                                  int(dtype_size))
    _need(n >= 0, "shape arguments must be positive")
    return n


def copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, pairs: torch.Tensor) -> None:
    """Copy-on-write on the device: block ``pairs[i, 1]`` of both pools
    becomes a copy of block ``pairs[i, 0]`` (``pairs`` int32 [n, 2] on the
    pools' device; bf16 or uint8 (FP8) pools)."""
    for c in (k_cache, v_cache):
        _need(c.is_cuda and c.is_contiguous() and c.dim() == 4 and
              c.dtype in (torch.bfloat16, torch.uint8),
              "pools must be contiguous bf16 or uint8 CUDA tensors [NB, bs, Hkv, d]")
    _need(k_cache.shape == v_cache.shape and k_cache.dtype == v_cache.dtype,
          "k_cache and v_cache differ")
    _need(pairs.dtype == torch.int32 and pairs.is_contiguous() and pairs.dim() == 2 and
          pairs.shape[1] == 2 and (pairs.numel() == 0 or pairs.device == k_cache.device),
          "pairs must be a contiguous int32 [n, 2] tensor on the pools' device")
    st = lib.pkv_copy_blocks(_ptr(k_cache), _ptr(v_cache), cache_desc(k_cache),
                             k_cache.element_size(), _ptr(pairs), pairs.shape[0],
                             _stream(k_cache))
    _check("pkv_copy_blocks", st)
