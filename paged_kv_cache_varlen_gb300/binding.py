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
    "pkv_lse_merge": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp]),
    "pkv_paged_attention_varlen_noalloc": (
        _i32, [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp] + [_i32] * 9
        + [ctypes.c_float, _i32, _vp, _vp]),
    "pkv_status_string": (ctypes.c_char_p, [_i32]),
    "pkv_abi_version": (_i32, []),
}

DEV_BAD_SLOT = 1
DEV_BAD_BLOCK = 2
DEV_BAD_LENGTHS = 4
DEV_TIMEOUT = 8


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
    st = load_library().pkv_paged_attention_varlen_noalloc(
        _ptr(out), _ptr(out_lse), _ptr(q), _ptr(kv_pool), _ptr(block_table),
        block_table.shape[1], _ptr(cu_seqlens), _ptr(seq_lens), b, t, int(max_query_len),
        int(max_seq_len), h, hkv, d, bs, nb, float(scale), int(partition_size),
        _ptr(dev_status), _stream(stream, q.device))
    _check(st, "paged_attention_varlen_noalloc")
    return out, out_lse
