"""Sequence parallelism over ranks: each rank attends to a key range of
every request and the pieces are merged by log-sum-exp.

Page 1 (从 token 调度到采样输出…), §07: long-context chunked prefill,
Flash-Decoding and sequence parallelism split the sequence dimension and
renormalise the pieces exactly with log-sum-exp. Here a request's context is
cut into contiguous, block-aligned key ranges, one per rank; every rank holds
the blocks of its own range in its own pool and runs
``pkv_paged_attention_varlen_range`` for all of the request's queries over
that range; the normalised pieces ``(out, lse)`` are exchanged (one
all-gather of ``T * H * (D + 1)`` floats per rank) and merged with
``pkv_lse_merge``.

This module only does the bookkeeping on the host (which keys a rank holds,
its shifted block table and positions) and the exchange; every arithmetic
step runs in the library's kernels. A rank that holds no key of a request
contributes an empty piece (out 0, lse -inf), which the merge ignores.
"""
from __future__ import annotations

import numpy as np


def key_ranges(total_len: int, world: int, block_size: int) -> list[tuple[int, int]]:
    """Contiguous key ranges [start, end) of one context, one per rank, cut at
    block boundaries and as even as whole blocks allow (ranks past the last
    block get an empty range)."""
    nblk = -(-int(total_len) // block_size)
    per, extra = divmod(nblk, world)
    out, b = [], 0
    for r in range(world):
        n = per + (1 if r < extra else 0)
        start = min(b * block_size, int(total_len))
        out.append((start, min((b + n) * block_size, int(total_len))))
        b += n
    return out


def shard_inputs(block_table: np.ndarray, seq_lens: np.ndarray, query_lens: np.ndarray,
                 rank: int, world: int, block_size: int) -> dict:
    """Inputs of this rank's range call for a batch (host int32 arrays).

    ``block_table``/``seq_lens``/``query_lens`` describe the whole contexts
    (lengths include the step's queries). Returns the requests this rank
    holds keys of (``keep``), their tables shifted to the rank's first block,
    their local key counts, the absolute position of their first key and of
    their first query, and the rank's ``(start, end)`` per request.
    """
    B = int(seq_lens.shape[0])
    keep, tables, lens, kstart, qstart, ranges = [], [], [], [], [], []
    width = 1
    for i in range(B):
        L, q = int(seq_lens[i]), int(query_lens[i])
        s, e = key_ranges(L, world, block_size)[rank]
        ranges.append((s, e))
        if e <= s:
            continue
        nb = -(-(e - s) // block_size)
        row = block_table[i, s // block_size:s // block_size + nb]
        keep.append(i)
        tables.append(row)
        lens.append(e - s)
        kstart.append(s)
        qstart.append(L - q)
        width = max(width, nb)
    table = np.full((max(len(keep), 1), width), -1, dtype=np.int32)
    for r, row in enumerate(tables):
        table[r, :row.shape[0]] = row
    return {"keep": np.array(keep, dtype=np.int64), "block_table": table[:len(keep)],
            "seq_lens": np.array(lens, dtype=np.int32),
            "key_start_pos": np.array(kstart, dtype=np.int32),
            "query_start_pos": np.array(qstart, dtype=np.int32), "ranges": ranges}


def compact_queries(cu_seqlens: np.ndarray, keep: np.ndarray):
    """Token indices and cu_seqlens of the kept requests' queries."""
    tok = [np.arange(cu_seqlens[i], cu_seqlens[i + 1]) for i in keep]
    tok = np.concatenate(tok).astype(np.int64) if tok else np.zeros(0, dtype=np.int64)
    ql = np.array([cu_seqlens[i + 1] - cu_seqlens[i] for i in keep], dtype=np.int64)
    cu = np.zeros(len(keep) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(ql)
    return tok, cu


def rank_piece(q, pool, block_table: np.ndarray, cu_seqlens: np.ndarray, seq_lens: np.ndarray,
               rank: int, world: int, scale: float, dev_status=None, partition_size: int = -1):
    """This rank's piece ``(out [T,H,D], lse [T,H])`` of attention over the
    whole batch, computed on the GPU from the keys of its range (``q`` and
    ``pool`` are device tensors; the tables are host arrays)."""
    import torch

    from . import binding as pkv

    T, H, D = q.shape
    bs = pool.shape[2]
    ql = np.diff(cu_seqlens).astype(np.int32)
    sh = shard_inputs(block_table, seq_lens, ql, rank, world, bs)
    out = torch.zeros((T, H, D), dtype=torch.float32, device=q.device)
    lse = torch.full((T, H), float("-inf"), dtype=torch.float32, device=q.device)
    if sh["keep"].size == 0:
        return out, lse
    tok, cu = compact_queries(cu_seqlens, sh["keep"])
    dev = q.device

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

    tok_t = torch.from_numpy(tok).to(dev)
    qk = q.index_select(0, tok_t).contiguous()
    o, ls = pkv.paged_attention_varlen_range(
        qk, pool, i32(sh["block_table"]), i32(cu), i32(sh["seq_lens"]),
        i32(sh["key_start_pos"]), i32(sh["query_start_pos"]), int(ql[sh["keep"]].max()),
        int(sh["seq_lens"].max()), out_lse=torch.empty((tok.shape[0], H), dtype=torch.float32,
                                                       device=dev),
        scale=scale, partition_size=partition_size, dev_status=dev_status)
    out.index_copy_(0, tok_t, o)
    lse.index_copy_(0, tok_t, ls)
    return out, lse


def gather_pieces(out, lse, group=None):
    """All-gather every rank's piece: returns ``(part_out [W,T,H,D],
    part_lse [W,T,H])`` on this rank's device. With a gloo group the exchange
    goes through host memory."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    host = dist.get_backend(group) == "gloo"
    o = out.cpu() if host else out
    ls = lse.cpu() if host else lse
    os_ = [torch.empty_like(o) for _ in range(world)]
    ls_ = [torch.empty_like(ls) for _ in range(world)]
    dist.all_gather(os_, o, group=group)
    dist.all_gather(ls_, ls, group=group)
    return (torch.stack(os_).to(out.device).contiguous(),
            torch.stack(ls_).to(out.device).contiguous())


def merge_pieces(part_out, part_lse):
    """Attention over the whole contexts from the ranks' pieces
    (``pkv_lse_merge`` on the GPU)."""
    from . import binding as pkv

    T, H = part_lse.shape[1:]
    import torch

    out_lse = torch.empty((T, H), dtype=torch.float32, device=part_out.device)
    return pkv.lse_merge(part_out, part_lse, out_lse=out_lse)
