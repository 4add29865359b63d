"""Host-side index checks for debugging (``PKV_DEBUG_CHECKS=1``).

The kernels check every index they read and report a bad one through a
status bit (``dev_status``), skipping the item; they cannot say which entry
was wrong, and no memory checker runs on the GPUs this library targets. With
the environment variable ``PKV_DEBUG_CHECKS=1`` the binding copies the index
tables of each call to the host first (synchronising the stream) and checks
every entry the kernels would read, raising ``ValueError`` with the first
offending one. This is bookkeeping on the tables only: no attention
arithmetic runs here, and the call itself still runs on the GPU.

What is checked follows the documented contracts of ``include/pkv.h``:
cu_seqlens_q non-decreasing from 0 to num_tokens; every request's query count
at most max_query_len; its context length at least its query count (or, for
key ranges, at least 1 with non-negative positions), at most max_seq_len and
within its table row; every block id a request's context covers inside the
pool; every slot of the KV write inside the pool (or -1, skipped); and, for
the combined KV write and attention call, every slot the one block_table gives
to its token's query position.
"""
from __future__ import annotations

import os

import numpy as np


def enabled() -> bool:
    return os.environ.get("PKV_DEBUG_CHECKS", "") == "1"


def _host(t) -> np.ndarray:
    if hasattr(t, "detach"):
        return t.detach().to("cpu").numpy()
    return np.asarray(t)


def check_attention_tables(cu_seqlens, seq_lens, block_table, *, num_tokens: int,
                           max_query_len: int, max_seq_len: int, num_blocks: int,
                           block_size: int, key_start=None, query_start=None) -> None:
    """Raise ValueError on the first entry the attention kernels would reject."""
    cu = _host(cu_seqlens).astype(np.int64)
    lens = _host(seq_lens).astype(np.int64)
    table = _host(block_table).astype(np.int64)
    b = lens.shape[0]
    if cu.shape[0] != b + 1 or table.shape[0] != b:
        raise ValueError(f"table shapes: cu_seqlens {cu.shape}, seq_lens {lens.shape}, "
                         f"block_table {table.shape}")
    if cu[0] != 0:
        raise ValueError(f"cu_seqlens_q[0] = {cu[0]}, not 0")
    if cu[b] != num_tokens:
        raise ValueError(f"cu_seqlens_q[{b}] = {cu[b]}, not num_tokens = {num_tokens}")
    qlen = np.diff(cu)
    bad = np.nonzero(qlen < 0)[0]
    if bad.size:
        i = int(bad[0])
        raise ValueError(f"cu_seqlens_q decreases at request {i}: {cu[i]} -> {cu[i + 1]}")
    bad = np.nonzero(qlen > max_query_len)[0]
    if bad.size:
        i = int(bad[0])
        raise ValueError(f"request {i} has {qlen[i]} queries > max_query_len {max_query_len}")
    ranged = key_start is not None
    if ranged:
        ks = _host(key_start).astype(np.int64)
        qs = _host(query_start).astype(np.int64)
        bad = np.nonzero((ks < 0) | (qs < 0))[0]
        if bad.size:
            i = int(bad[0])
            raise ValueError(f"request {i}: key_start {ks[i]} / query_start {qs[i]} negative")
        bad = np.nonzero((lens < 1) & (qlen > 0))[0]
    else:
        bad = np.nonzero(lens < qlen)[0]
    if bad.size:
        i = int(bad[0])
        raise ValueError(f"request {i}: seq_len {lens[i]} shorter than its {qlen[i]} queries")
    bad = np.nonzero(lens > max_seq_len)[0]
    if bad.size:
        i = int(bad[0])
        raise ValueError(f"request {i}: seq_len {lens[i]} > max_seq_len {max_seq_len}")
    nblk = -(-lens // block_size)
    bad = np.nonzero(nblk > table.shape[1])[0]
    if bad.size:
        i = int(bad[0])
        raise ValueError(f"request {i}: seq_len {lens[i]} needs {nblk[i]} blocks, its table "
                         f"row holds {table.shape[1]}")
    for i in range(b):
        if qlen[i] == 0:
            continue
        ids = table[i, :nblk[i]]
        out = np.nonzero((ids < 0) | (ids >= num_blocks))[0]
        if out.size:
            j = int(out[0])
            raise ValueError(f"request {i}: block_table[{i}][{j}] = {ids[j]} outside the pool "
                             f"[0, {num_blocks})")


def check_append_slots(cu_seqlens, seq_lens, block_table, slot_mapping, *,
                       block_size: int) -> None:
    """For the combined KV write and attention call: raise ValueError unless
    every token's slot (-1: skipped) is the pool slot block_table gives to the
    token's position, seq_len - query_len + j for its request's query j."""
    cu = _host(cu_seqlens).astype(np.int64)
    lens = _host(seq_lens).astype(np.int64)
    table = _host(block_table).astype(np.int64)
    slots = _host(slot_mapping).astype(np.int64)
    qlen = np.diff(cu)
    req = np.repeat(np.arange(lens.shape[0]), qlen)
    pos = lens[req] - qlen[req] + (np.arange(cu[-1]) - cu[req])
    want = table[req, pos // block_size] * block_size + pos % block_size
    bad = np.nonzero((slots != -1) & (slots != want))[0]
    if bad.size:
        t = int(bad[0])
        raise ValueError(f"slot_mapping[{t}] = {slots[t]}: request {int(req[t])}'s position "
                         f"{int(pos[t])} is slot {int(want[t])}")


def check_slot_mapping(slot_mapping, *, num_blocks: int, block_size: int) -> None:
    """Raise ValueError on the first slot outside the pool (-1 is skipped)."""
    slots = _host(slot_mapping).astype(np.int64)
    bad = np.nonzero((slots < -1) | (slots >= num_blocks * block_size))[0]
    if bad.size:
        t = int(bad[0])
        raise ValueError(f"slot_mapping[{t}] = {slots[t]} outside the pool "
                         f"[0, {num_blocks * block_size}) and not -1")
