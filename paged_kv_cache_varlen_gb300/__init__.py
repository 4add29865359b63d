"""Paged KV-cache attention for GB300 (sm_103a).

The compute lives in ``libpkv.so`` (hand-written CUDA behind a C ABI, see
``include/pkv.h``); :mod:`.binding` marshals torch tensors into it. The
library is loaded on first use and its absence is an error: there is no CPU
fallback.
"""
from .binding import (  # noqa: F401
    PkvError,
    attention_workspace_size,
    kv_cache_write,
    library_path,
    lse_merge,
    paged_attention_varlen,
    paged_attention_varlen_append,
    paged_attention_varlen_range,
)

__all__ = [
    "PkvError",
    "attention_workspace_size",
    "kv_cache_write",
    "library_path",
    "lse_merge",
    "paged_attention_varlen",
    "paged_attention_varlen_append",
    "paged_attention_varlen_range",
]
