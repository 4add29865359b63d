"""Reference block manager for the paged KV cache (test infrastructure).

This module is TEST INFRASTRUCTURE, like the rest of ``oracle/``: only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import it. It is the plain, slow statement of what the host-side allocator of
the paged cache does, written from page 2 (su666666.com, "PagedAttention
deep-dive", the block-table and copy-on-write passages):

* the physical block pool is carved up once at start-up; free blocks wait in
  a pool;
* every sequence owns a block table mapping its logical blocks, in order, to
  physical blocks; logical token ``p`` lives in slot
  ``table[p // block_size] * block_size + p % block_size``;
* when a sequence needs room for a new token and its last block is full (or
  it has none), the scheduler takes a free block from the pool and appends it
  to the sequence's table;
* forking a sequence (one prompt, several candidate continuations) copies only
  the block table: parent and child point at the same physical blocks;
* a shared block gets its own copy only when a sequence writes into it:
  "write-time allocation" of a new block for the sequence that diverges.

Readings where the page is silent:

* free-pool order: first in, first out, starting from ``free_order`` (default
  ascending ids); a released block joins the back of the queue;
* a shared block is copied only when the writer's next token falls inside it
  (the block is partially filled); a full shared block is never written again,
  so the next token simply goes to a fresh block, with no copy;
* the copy is of the whole block (all ``block_size`` slots of K and V), source
  block to destination block, executed on the GPU before the step's KV write;
* an append that cannot be satisfied from the pool raises ``OutOfBlocks`` and
  changes nothing.
"""
from __future__ import annotations

from collections import deque


class OutOfBlocks(RuntimeError):
    pass


class BlockManagerOracle:
    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of the block ids")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free = deque(order)
        self.ref = [0] * num_blocks
        self.tables: dict[int, list[int]] = {}
        self.lens: dict[int, int] = {}

    # -- sequences -----------------------------------------------------------
    def add_seq(self, sid: int) -> None:
        if sid in self.tables:
            raise KeyError(f"sequence {sid} exists")
        self.tables[sid] = []
        self.lens[sid] = 0

    def fork(self, parent: int, child: int) -> None:
        """The child gets a copy of the parent's block table (and length);
        every block it names gains one more reference."""
        if parent not in self.tables or child in self.tables:
            raise KeyError("unknown parent or existing child")
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for b in self.tables[child]:
            self.ref[b] += 1

    def free_seq(self, sid: int) -> None:
        for b in self.tables.pop(sid):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.append(b)
        del self.lens[sid]

    # -- growth --------------------------------------------------------------
    def blocks_needed(self, sid: int, n: int) -> int:
        """Free blocks an append of n tokens takes: one per new logical block,
        plus one for copying a shared, partially filled last block."""
        length, bs = self.lens[sid], self.block_size
        need = 0
        if n > 0 and length % bs != 0 and self.ref[self.tables[sid][-1]] > 1:
            need += 1
        first_new = -(-length // bs)          # logical blocks already present
        last = (length + n - 1) // bs if n > 0 else first_new - 1
        need += max(0, last + 1 - first_new)
        return need

    def append(self, sid: int, n: int):
        """Room for n new tokens. Returns (slots, copies): the slot of every
        new token in order, and the (src, dst) block copies to run first."""
        if sid not in self.tables:
            raise KeyError(f"unknown sequence {sid}")
        if n < 0:
            raise ValueError("negative token count")
        if self.blocks_needed(sid, n) > len(self.free):
            raise OutOfBlocks(f"sequence {sid} needs more blocks than are free")
        table, bs = self.tables[sid], self.block_size
        slots, copies = [], []
        for _ in range(n):
            pos = self.lens[sid]
            logical, offset = divmod(pos, bs)
            if offset == 0:
                blk = self.free.popleft()
                self.ref[blk] = 1
                table.append(blk)
            elif self.ref[table[logical]] > 1:
                old = table[logical]
                blk = self.free.popleft()
                self.ref[blk] = 1
                self.ref[old] -= 1
                table[logical] = blk
                copies.append((old, blk))
            slots.append(table[logical] * bs + offset)
            self.lens[sid] = pos + 1
        return slots, copies

    # -- views ---------------------------------------------------------------
    def block_table(self, sid: int) -> list[int]:
        return list(self.tables[sid])

    def seq_len(self, sid: int) -> int:
        return self.lens[sid]

    def num_free(self) -> int:
        return len(self.free)

    def slot_of(self, sid: int, pos: int) -> int:
        table, bs = self.tables[sid], self.block_size
        return table[pos // bs] * bs + pos % bs


def apply_copies(pool, copies):
    """The block copies on a numpy pool [2, NB, BS, Hkv, D]: K and V of each
    destination block become those of its source (in order)."""
    out = pool.copy()
    for src, dst in copies:
        out[:, dst] = out[:, src]
    return out
