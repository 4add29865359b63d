"""Python binding of ``libpkv.so`` (argument marshalling only).

Every function here has the name of the C entry point without its ``pkv_``
prefix (``include/pkv.h``). It checks that the torch tensors have the dtype,
device and dense layout the C ABI expects, passes their device pointers and
the current CUDA stream, and raises :class:`PkvError` on a non-zero status.
All computation happens in the CUDA kernels behind the C ABI; if the library
is missing, the call fails: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import debug_checks

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(_HERE, "libpkv.so")

_lock = threading.Lock()
_handle = None

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32

# name -> (restype, argtypes), mirroring include/pkv.h
_SIGNATURES = {
    "pkv_kv_cache_write": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp]),
    "pkv_attention_workspace_size": (ctypes.c_size_t, [_i32] * 7),
    "pkv_paged_attention_varlen": (
        _i32, [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp] + [_i32] * 9
        + [ctypes.c_float, _i32, _vp, ctypes.c_size_t, _vp, _vp]),
    "pkv_paged_attention_varlen_append": (
        _i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp] + [_i32] * 9
        + [ctypes.c_float, _i32, _vp, ctypes.c_size_t, _vp, _vp]),
    "pkv_paged_attention_varlen_range": (
        _i32, [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp] + [_i32] * 9
        + [ctypes.c_float, _i32, _vp, ctypes.c_size_t, _vp, _vp]),
    "pkv_lse_merge": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp]),
    "pkv_paged_attention_varlen_noalloc": (
        _i32, [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp] + [_i32] * 9
        + [ctypes.c_float, _i32, _vp, _vp]),
    "pkv_cascade_workspace_size": (ctypes.c_size_t, [_i32] * 8),
    "pkv_cascade_decode": (
        _i32, [_vp, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _i32, _vp, _i32]
        + [_i32] * 6 + [ctypes.c_float, _vp, ctypes.c_size_t, _vp, _vp]),
    "pkv_copy_blocks": (_i32, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp]),
    "pkv_bm_create": (_i32, [_i32, _i32, _vp, ctypes.POINTER(_vp)]),
    "pkv_bm_destroy": (None, [_vp]),
    "pkv_bm_add_seq": (_i32, [_vp, ctypes.c_int64]),
    "pkv_bm_fork": (_i32, [_vp, ctypes.c_int64, ctypes.c_int64]),
    "pkv_bm_free_seq": (_i32, [_vp, ctypes.c_int64]),
    "pkv_bm_append": (_i32, [_vp, ctypes.c_int64, _i32, _vp, _vp, _vp, _i32, _vp]),
    "pkv_bm_build_step": (_i32, [_vp, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _i32,
                                 _vp]),
    "pkv_bm_num_free": (_i32, [_vp]),
    "pkv_bm_seq_len": (ctypes.c_int64, [_vp, ctypes.c_int64]),
    "pkv_bm_refcount": (_i32, [_vp, _i32]),
    "pkv_bm_block_table": (_i32, [_vp, ctypes.c_int64, _vp, _i32, _vp]),
    "pkv_status_string": (ctypes.c_char_p, [_i32]),
    "pkv_abi_version": (_i32, []),
}

DEV_BAD_SLOT = 1
DEV_BAD_BLOCK = 2
DEV_BAD_LENGTHS = 4
DEV_TIMEOUT = 8
DEV_V_RANGE = 16


class PkvError(RuntimeError):
    """A libpkv call returned an error status (or the library is missing)."""

    def __init__(self, message: str, status: int | None = None):
        super().__init__(message)
        self.status = status


def library_path() -> str:
    return LIBRARY


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load ``libpkv.so`` once and declare the C signatures."""
    global _handle
    with _lock:
        if _handle is not None and path is None:
            return _handle
        p = path or LIBRARY
        if not os.path.exists(p):
            raise PkvError(
                f"{p} is missing: build it first (python -c 'import __graft_entry__ as g; "
                "g.build()'). There is no CPU fallback.")
        lib = ctypes.CDLL(p)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _handle = lib
        return lib


def _check(status: int, what: str) -> None:
    if status != 0:
        msg = load_library().pkv_status_string(status).decode()
        raise PkvError(f"{what}: {msg} (status {status})", status)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _need(t: torch.Tensor, dtype, ndim: int, name: str) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def kv_cache_write(kv_pool: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                   slot_mapping: torch.Tensor, dev_status: torch.Tensor | None = None,
                   stream=None) -> None:
    """Scatter k_new/v_new [T,Hkv,D] bf16 into kv_pool [2,NB,BS,Hkv,D] bf16."""
    _need(kv_pool, torch.bfloat16, 5, "kv_pool")
    _need(k_new, torch.bfloat16, 3, "k_new")
    _need(v_new, torch.bfloat16, 3, "v_new")
    _need(slot_mapping, torch.int32, 1, "slot_mapping")
    _, nb, bs, hkv, d = kv_pool.shape
    t = slot_mapping.shape[0]
    if tuple(k_new.shape) != (t, hkv, d) or tuple(v_new.shape) != (t, hkv, d):
        raise ValueError("k_new / v_new must be [num_tokens, num_kv_heads, head_dim]")
    if dev_status is not None:
        _need(dev_status, torch.int32, 1, "dev_status")
    if debug_checks.enabled():
        debug_checks.check_slot_mapping(slot_mapping, num_blocks=nb, block_size=bs)
    st = load_library().pkv_kv_cache_write(
        _ptr(kv_pool), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), t, nb, bs, hkv, d,
        _ptr(dev_status), _stream(stream, kv_pool.device))
    _check(st, "kv_cache_write")


def attention_workspace_size(num_seqs: int, num_tokens: int, num_heads: int, num_kv_heads: int,
                             head_dim: int, max_seq_len: int, partition_size: int = -1) -> int:
    return int(load_library().pkv_attention_workspace_size(
        num_seqs, num_tokens, num_heads, num_kv_heads, head_dim, max_seq_len, partition_size))


def paged_attention_varlen(q: torch.Tensor, kv_pool: torch.Tensor, block_table: torch.Tensor,
                           cu_seqlens: torch.Tensor, seq_lens: torch.Tensor,
                           max_query_len: int, max_seq_len: int, *,
                           out: torch.Tensor | None = None, out_lse: torch.Tensor | None = None,
                           scale: float | None = None, partition_size: int = -1,
                           workspace: torch.Tensor | None = None,
                           dev_status: torch.Tensor | None = None, stream=None):
    """Causal GQA attention of q [T,H,D] bf16 over the paged pool.

    Returns ``(out, out_lse)``; ``out`` is fp32 [T,H,D], ``out_lse`` fp32
    [T,H] or None. Missing ``out`` / ``workspace`` buffers are allocated with
    torch (the library itself never allocates); a workspace passed in must
    have been zero-filled before its first use (``attention_workspace_size``).
    """
    _need(q, torch.bfloat16, 3, "q")
    _need(kv_pool, torch.bfloat16, 5, "kv_pool")
    _need(block_table, torch.int32, 2, "block_table")
    _need(cu_seqlens, torch.int32, 1, "cu_seqlens")
    _need(seq_lens, torch.int32, 1, "seq_lens")
    t, h, d = q.shape
    _, nb, bs, hkv, d2 = kv_pool.shape
    if d2 != d:
        raise ValueError("q and kv_pool head_dim differ")
    b = seq_lens.shape[0]
    if cu_seqlens.shape[0] != b + 1 or block_table.shape[0] != b:
        raise ValueError("cu_seqlens must be [B+1] and block_table [B, max_blocks]")
    if out is None:
        out = torch.empty((t, h, d), dtype=torch.float32, device=q.device)
    _need(out, torch.float32, 3, "out")
    if out_lse is not None:
        _need(out_lse, torch.float32, 2, "out_lse")
    if dev_status is not None:
        _need(dev_status, torch.int32, 1, "dev_status")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if debug_checks.enabled():
        debug_checks.check_attention_tables(
            cu_seqlens, seq_lens, block_table, num_tokens=t, max_query_len=int(max_query_len),
            max_seq_len=int(max_seq_len), num_blocks=nb, block_size=bs)
    need = attention_workspace_size(b, t, h, hkv, d, max_seq_len, partition_size)
    if need and workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load_library().pkv_paged_attention_varlen(
        _ptr(out), _ptr(out_lse), _ptr(q), _ptr(kv_pool), _ptr(block_table),
        block_table.shape[1], _ptr(cu_seqlens), _ptr(seq_lens), b, t, int(max_query_len),
        int(max_seq_len), h, hkv, d, bs, nb, float(scale), int(partition_size),
        _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream, q.device))
    _check(st, "paged_attention_varlen")
    return out, out_lse


def paged_attention_varlen_append(q: torch.Tensor, kv_pool: torch.Tensor, k_new: torch.Tensor,
                                  v_new: torch.Tensor, slot_mapping: torch.Tensor,
                                  block_table: torch.Tensor, cu_seqlens: torch.Tensor,
                                  seq_lens: torch.Tensor, max_query_len: int, max_seq_len: int, *,
                                  out: torch.Tensor | None = None,
                                  out_lse: torch.Tensor | None = None, scale: float | None = None,
                                  partition_size: int = -1, workspace: torch.Tensor | None = None,
                                  dev_status: torch.Tensor | None = None, stream=None):
    """A step's KV write and attention in one call (``kv_cache_write`` then
    ``paged_attention_varlen``, overlapped). ``slot_mapping[t]`` must be the
    pool slot ``block_table`` gives to token t's position (the step's
    appended slots). Returns ``(out, out_lse)`` as ``paged_attention_varlen``."""
    _need(q, torch.bfloat16, 3, "q")
    _need(kv_pool, torch.bfloat16, 5, "kv_pool")
    _need(k_new, torch.bfloat16, 3, "k_new")
    _need(v_new, torch.bfloat16, 3, "v_new")
    _need(slot_mapping, torch.int32, 1, "slot_mapping")
    _need(block_table, torch.int32, 2, "block_table")
    _need(cu_seqlens, torch.int32, 1, "cu_seqlens")
    _need(seq_lens, torch.int32, 1, "seq_lens")
    t, h, d = q.shape
    _, nb, bs, hkv, d2 = kv_pool.shape
    if d2 != d:
        raise ValueError("q and kv_pool head_dim differ")
    if slot_mapping.shape[0] != t or tuple(k_new.shape) != (t, hkv, d) or \
            tuple(v_new.shape) != (t, hkv, d):
        raise ValueError("k_new / v_new must be [num_tokens, num_kv_heads, head_dim] and "
                         "slot_mapping [num_tokens]")
    b = seq_lens.shape[0]
    if cu_seqlens.shape[0] != b + 1 or block_table.shape[0] != b:
        raise ValueError("cu_seqlens must be [B+1] and block_table [B, max_blocks]")
    if out is None:
        out = torch.empty((t, h, d), dtype=torch.float32, device=q.device)
    _need(out, torch.float32, 3, "out")
    if out_lse is not None:
        _need(out_lse, torch.float32, 2, "out_lse")
    if dev_status is not None:
        _need(dev_status, torch.int32, 1, "dev_status")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if debug_checks.enabled():
        debug_checks.check_slot_mapping(slot_mapping, num_blocks=nb, block_size=bs)
        debug_checks.check_attention_tables(
            cu_seqlens, seq_lens, block_table, num_tokens=t, max_query_len=int(max_query_len),
            max_seq_len=int(max_seq_len), num_blocks=nb, block_size=bs)
        debug_checks.check_append_slots(cu_seqlens, seq_lens, block_table, slot_mapping,
                                        block_size=bs)
    need = attention_workspace_size(b, t, h, hkv, d, max_seq_len, partition_size)
    if need and workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load_library().pkv_paged_attention_varlen_append(
        _ptr(out), _ptr(out_lse), _ptr(q), _ptr(kv_pool), _ptr(k_new), _ptr(v_new),
        _ptr(slot_mapping), _ptr(block_table), block_table.shape[1], _ptr(cu_seqlens),
        _ptr(seq_lens), b, t, int(max_query_len), int(max_seq_len), h, hkv, d, bs, nb,
        float(scale), int(partition_size), _ptr(workspace), ws_bytes, _ptr(dev_status),
        _stream(stream, q.device))
    _check(st, "paged_attention_varlen_append")
    return out, out_lse


def paged_attention_varlen_range(q: torch.Tensor, kv_pool: torch.Tensor,
                                 block_table: torch.Tensor, cu_seqlens: torch.Tensor,
                                 seq_lens: torch.Tensor, key_start_pos: torch.Tensor,
                                 query_start_pos: torch.Tensor, max_query_len: int,
                                 max_seq_len: int, *, out: torch.Tensor | None = None,
                                 out_lse: torch.Tensor | None = None, scale: float | None = None,
                                 partition_size: int = -1, workspace: torch.Tensor | None = None,
                                 dev_status: torch.Tensor | None = None, stream=None):
    """Attention over a range of each request's keys (``pkv_paged_attention_varlen_range``).

    Request i's table holds ``seq_lens[i]`` keys at absolute positions
    ``key_start_pos[i] + p``; its queries sit at ``query_start_pos[i] + j``
    and see the keys at or before their own position. Returns the normalised
    piece ``(out, out_lse)``; pieces of one context merge with :func:`lse_merge`.
    """
    _need(q, torch.bfloat16, 3, "q")
    _need(kv_pool, torch.bfloat16, 5, "kv_pool")
    _need(block_table, torch.int32, 2, "block_table")
    for t, name in ((cu_seqlens, "cu_seqlens"), (seq_lens, "seq_lens"),
                    (key_start_pos, "key_start_pos"), (query_start_pos, "query_start_pos")):
        _need(t, torch.int32, 1, name)
    t, h, d = q.shape
    _, nb, bs, hkv, d2 = kv_pool.shape
    if d2 != d:
        raise ValueError("q and kv_pool head_dim differ")
    b = seq_lens.shape[0]
    if (cu_seqlens.shape[0] != b + 1 or block_table.shape[0] != b
            or key_start_pos.shape[0] != b or query_start_pos.shape[0] != b):
        raise ValueError("cu_seqlens must be [B+1]; block_table, key_start_pos and "
                         "query_start_pos one row per request")
    if out is None:
        out = torch.empty((t, h, d), dtype=torch.float32, device=q.device)
    _need(out, torch.float32, 3, "out")
    if out_lse is not None:
        _need(out_lse, torch.float32, 2, "out_lse")
    if dev_status is not None:
        _need(dev_status, torch.int32, 1, "dev_status")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if debug_checks.enabled():
        debug_checks.check_attention_tables(
            cu_seqlens, seq_lens, block_table, num_tokens=t, max_query_len=int(max_query_len),
            max_seq_len=int(max_seq_len), num_blocks=nb, block_size=bs,
            key_start=key_start_pos, query_start=query_start_pos)
    need = attention_workspace_size(b, t, h, hkv, d, max_seq_len, partition_size)
    if need and workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load_library().pkv_paged_attention_varlen_range(
        _ptr(out), _ptr(out_lse), _ptr(q), _ptr(kv_pool), _ptr(block_table),
        block_table.shape[1], _ptr(cu_seqlens), _ptr(seq_lens), _ptr(key_start_pos),
        _ptr(query_start_pos), b, t, int(max_query_len), int(max_seq_len), h, hkv, d, bs, nb,
        float(scale), int(partition_size), _ptr(workspace), ws_bytes, _ptr(dev_status),
        _stream(stream, q.device))
    _check(st, "paged_attention_varlen_range")
    return out, out_lse


def lse_merge(part_out: torch.Tensor, part_lse: torch.Tensor, *,
              out: torch.Tensor | None = None, out_lse: torch.Tensor | None = None,
              stream=None):
    """Merge part_out [P,T,H,D] / part_lse [P,T,H] fp32 into out [T,H,D]."""
    _need(part_out, torch.float32, 4, "part_out")
    _need(part_lse, torch.float32, 3, "part_lse")
    p, t, h, d = part_out.shape
    if tuple(part_lse.shape) != (p, t, h):
        raise ValueError("part_lse must be [P, T, H]")
    if out is None:
        out = torch.empty((t, h, d), dtype=torch.float32, device=part_out.device)
    _need(out, torch.float32, 3, "out")
    if out_lse is not None:
        _need(out_lse, torch.float32, 2, "out_lse")
    st = load_library().pkv_lse_merge(_ptr(out), _ptr(out_lse), _ptr(part_out), _ptr(part_lse),
                                      p, t, h, d, _stream(stream, part_out.device))
    _check(st, "lse_merge")
    return out, out_lse


def paged_attention_varlen_noalloc(q: torch.Tensor, kv_pool: torch.Tensor,
                                   block_table: torch.Tensor, cu_seqlens: torch.Tensor,
                                   seq_lens: torch.Tensor, max_query_len: int, max_seq_len: int,
                                   *, out: torch.Tensor, out_lse: torch.Tensor | None = None,
                                   scale: float | None = None, partition_size: int = -1,
                                   dev_status: torch.Tensor | None = None, stream=None):
    """:func:`paged_attention_varlen` for callers that cannot allocate.

    For code that may not allocate device memory (its memory manager owns
    the GPU, or it is not allowed to call cudaMalloc while serving): the
    split-KV scratch comes from a fixed 16 MiB array inside the library, so
    nothing is allocated here and ``out`` must be passed in. Raises
    :class:`PkvError` (status 4) when the sizes need more scratch than that.
    Calls that may overlap on the GPU share the array and race.
    """
    _need(q, torch.bfloat16, 3, "q")
    _need(kv_pool, torch.bfloat16, 5, "kv_pool")
    _need(block_table, torch.int32, 2, "block_table")
    _need(cu_seqlens, torch.int32, 1, "cu_seqlens")
    _need(seq_lens, torch.int32, 1, "seq_lens")
    _need(out, torch.float32, 3, "out")
    t, h, d = q.shape
    _, nb, bs, hkv, d2 = kv_pool.shape
    if d2 != d:
        raise ValueError("q and kv_pool head_dim differ")
    b = seq_lens.shape[0]
    if cu_seqlens.shape[0] != b + 1 or block_table.shape[0] != b:
        raise ValueError("cu_seqlens must be [B+1] and block_table [B, max_blocks]")
    if out_lse is not None:
        _need(out_lse, torch.float32, 2, "out_lse")
    if dev_status is not None:
        _need(dev_status, torch.int32, 1, "dev_status")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if debug_checks.enabled():
        debug_checks.check_attention_tables(
            cu_seqlens, seq_lens, block_table, num_tokens=t, max_query_len=int(max_query_len),
            max_seq_len=int(max_seq_len), num_blocks=nb, block_size=bs)
    st = load_library().pkv_paged_attention_varlen_noalloc(
        _ptr(out), _ptr(out_lse), _ptr(q), _ptr(kv_pool), _ptr(block_table),
        block_table.shape[1], _ptr(cu_seqlens), _ptr(seq_lens), b, t, int(max_query_len),
        int(max_seq_len), h, hkv, d, bs, nb, float(scale), int(partition_size),
        _ptr(dev_status), _stream(stream, q.device))
    _check(st, "paged_attention_varlen_noalloc")
    return out, out_lse


def copy_blocks(kv_pool: torch.Tensor, copy_src: torch.Tensor, copy_dst: torch.Tensor, *,
                dev_status: torch.Tensor | None = None, stream=None) -> None:
    """Whole-block copies inside the pool (device int32 ``copy_src``/``copy_dst``),
    the device half of copy-on-write; run before the step's KV write."""
    _need(kv_pool, torch.bfloat16, 5, "kv_pool")
    _need(copy_src, torch.int32, 1, "copy_src")
    _need(copy_dst, torch.int32, 1, "copy_dst")
    if copy_src.shape != copy_dst.shape:
        raise ValueError("copy_src and copy_dst differ in length")
    if dev_status is not None:
        _need(dev_status, torch.int32, 1, "dev_status")
    _, nb, bs, hkv, d = kv_pool.shape
    st = load_library().pkv_copy_blocks(
        _ptr(kv_pool), _ptr(copy_src), _ptr(copy_dst), copy_src.shape[0], nb, bs, hkv, d,
        _ptr(dev_status), _stream(stream, kv_pool.device))
    _check(st, "copy_blocks")


class BlockManager:
    """The host block manager of ``libpkv`` (native C++ behind the C ABI):
    free pool, per-sequence block tables, fork and copy-on-write."""

    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        import numpy as np

        self._np = np
        lib = load_library()
        h = _vp()
        order = None
        if free_order is not None:
            order = np.ascontiguousarray(free_order, dtype=np.int32)
            if order.shape != (num_blocks,):
                raise ValueError("free_order must hold every block id once")
        st = lib.pkv_bm_create(num_blocks, block_size,
                               order.ctypes.data if order is not None else None, ctypes.byref(h))
        _check(st, "bm_create")
        self._lib, self._h = lib, h
        self.num_blocks, self.block_size = num_blocks, block_size

    def close(self):
        if self._h:
            self._lib.pkv_bm_destroy(self._h)
            self._h = _vp()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add_seq(self, seq_id: int):
        _check(self._lib.pkv_bm_add_seq(self._h, seq_id), "bm_add_seq")

    def fork(self, parent: int, child: int):
        _check(self._lib.pkv_bm_fork(self._h, parent, child), "bm_fork")

    def free_seq(self, seq_id: int):
        _check(self._lib.pkv_bm_free_seq(self._h, seq_id), "bm_free_seq")

    def append(self, seq_id: int, num_tokens: int):
        """Returns (slots, copies) like the reference manager."""
        np = self._np
        slots = np.zeros(max(num_tokens, 1), dtype=np.int32)
        src = np.zeros(1, dtype=np.int32)
        dst = np.zeros(1, dtype=np.int32)
        n = ctypes.c_int32(0)
        st = self._lib.pkv_bm_append(self._h, seq_id, num_tokens, slots.ctypes.data,
                                     src.ctypes.data, dst.ctypes.data, 1, ctypes.byref(n))
        _check(st, "bm_append")
        return slots[:num_tokens].tolist(), list(zip(src[:n.value].tolist(), dst[:n.value].tolist()))

    def build_step(self, seq_ids, num_new, max_blocks: int):
        """One batch: (block_table, seq_lens, cu_seqlens, slot_mapping, copy_src, copy_dst)
        as numpy int32 arrays, ready to be copied to the device."""
        np = self._np
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        nn = np.ascontiguousarray(num_new, dtype=np.int32)
        b = ids.shape[0]
        table = np.full((max(b, 1), max_blocks), -1, dtype=np.int32)
        lens = np.zeros(max(b, 1), dtype=np.int32)
        cu = np.zeros(b + 1, dtype=np.int32)
        slots = np.zeros(max(int(nn.sum()), 1), dtype=np.int32)
        cap = max(b, 1)
        src = np.zeros(cap, dtype=np.int32)
        dst = np.zeros(cap, dtype=np.int32)
        n = ctypes.c_int32(0)
        st = self._lib.pkv_bm_build_step(
            self._h, ids.ctypes.data, nn.ctypes.data, b, max_blocks, table.ctypes.data,
            lens.ctypes.data, cu.ctypes.data, slots.ctypes.data, src.ctypes.data, dst.ctypes.data,
            cap, ctypes.byref(n))
        _check(st, "bm_build_step")
        return (table[:b], lens[:b], cu, slots[:int(nn.sum())], src[:n.value], dst[:n.value])

    def num_free(self) -> int:
        return int(self._lib.pkv_bm_num_free(self._h))

    def seq_len(self, seq_id: int) -> int:
        return int(self._lib.pkv_bm_seq_len(self._h, seq_id))

    def refcount(self, block: int) -> int:
        return int(self._lib.pkv_bm_refcount(self._h, block))

    def block_table(self, seq_id: int):
        np = self._np
        n = ctypes.c_int32(0)
        cap = max(self.num_blocks, 1)
        out = np.zeros(cap, dtype=np.int32)
        st = self._lib.pkv_bm_block_table(self._h, seq_id, out.ctypes.data, cap, ctypes.byref(n))
        _check(st, "bm_block_table")
        return out[:n.value].tolist()


def cascade_workspace_size(num_seqs: int, num_prefix_groups: int, max_group_size: int,
                           max_prefix_len: int, max_tail_len: int, num_heads: int,
                           num_kv_heads: int, head_dim: int) -> int:
    return int(load_library().pkv_cascade_workspace_size(
        num_seqs, num_prefix_groups, max_group_size, max_prefix_len, max_tail_len, num_heads,
        num_kv_heads, head_dim))


def cascade_decode(q: torch.Tensor, kv_pool: torch.Tensor, group_starts: torch.Tensor,
                   prefix_lens: torch.Tensor, prefix_tables: torch.Tensor, max_group_size: int,
                   max_prefix_len: int, tail_tables: torch.Tensor, tail_lens: torch.Tensor,
                   max_tail_len: int, *, out: torch.Tensor | None = None,
                   out_lse: torch.Tensor | None = None, scale: float | None = None,
                   workspace: torch.Tensor | None = None, dev_status: torch.Tensor | None = None,
                   stream=None):
    """Decode attention with copy-on-write prefixes read once per group
    (see ``pkv_cascade_decode``). Allocates a zeroed workspace when none is given."""
    _need(q, torch.bfloat16, 3, "q")
    _need(kv_pool, torch.bfloat16, 5, "kv_pool")
    for t, name in ((group_starts, "group_starts"), (prefix_lens, "prefix_lens"),
                    (tail_lens, "tail_lens")):
        _need(t, torch.int32, 1, name)
    _need(prefix_tables, torch.int32, 2, "prefix_tables")
    _need(tail_tables, torch.int32, 2, "tail_tables")
    b, h, d = q.shape
    _, nb, bs, hkv, d2 = kv_pool.shape
    if d2 != d:
        raise ValueError("q and kv_pool head_dim differ")
    g = prefix_lens.shape[0]
    if group_starts.shape[0] != g + 1 or prefix_tables.shape[0] != g:
        raise ValueError("group_starts must be [G+1] and prefix_tables [G, max_prefix_blocks]")
    if tail_tables.shape[0] != b or tail_lens.shape[0] != b:
        raise ValueError("tail_tables and tail_lens must have one row per request")
    if out is None:
        out = torch.empty((b, h, d), dtype=torch.float32, device=q.device)
    _need(out, torch.float32, 3, "out")
    if out_lse is not None:
        _need(out_lse, torch.float32, 2, "out_lse")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = cascade_workspace_size(b, g, int(max_group_size), int(max_prefix_len),
                                  int(max_tail_len), h, hkv, d)
    if workspace is None:
        workspace = torch.zeros(max(need, 1), dtype=torch.uint8, device=q.device)
    st = load_library().pkv_cascade_decode(
        _ptr(out), _ptr(out_lse), _ptr(q), _ptr(kv_pool), g, _ptr(group_starts), _ptr(prefix_lens),
        _ptr(prefix_tables), prefix_tables.shape[1], int(max_group_size), int(max_prefix_len),
        _ptr(tail_tables), tail_tables.shape[1], _ptr(tail_lens), int(max_tail_len), b, h, hkv, d,
        bs, nb, float(scale), _ptr(workspace), workspace.numel(), _ptr(dev_status),
        _stream(stream, q.device))
    _check(st, "cascade_decode")
    return out, out_lse
