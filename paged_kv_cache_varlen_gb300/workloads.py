"""Seeded synthetic inputs for paged KV-cache attention.

This module plays the host scheduler and nothing more: it draws context and
query lengths, hands out physical blocks from a shuffled free list, builds the
per-request block tables, the flattened ``cu_seqlens`` and the ``slot_mapping``
of the new tokens, and fills the KV pool and Q/K/V with bf16 values. It holds
none of the attention arithmetic, so both the GPU path and the CPU oracle can
consume its arrays.

Recipe (numpy PCG64, ``default_rng(seed)``):

* lengths are integers drawn uniformly, both ends inclusive;
* physical block ids come from ``rng.permutation(num_blocks)``, consumed in
  order (shared prefix blocks are taken once per group);
* Q, new K/V and the pool are N(0,1) fp32 rounded to bf16 (round to nearest,
  ties to even); the pool is drawn from a child generator, in chunks;
* pool slots that hold no context token (never-used slots and the slots the
  step's own tokens will be written to) are poisoned with bf16 NaN (0x7FC0)
  in parity inputs, or set to zero for benchmark inputs.

The pool has the layout of one layer, ``[2, num_blocks, block_size,
num_kv_heads, head_dim]`` (K at index 0, V at index 1), and holds
``ceil(pool_factor * sum_i ceil(L_i / block_size))`` blocks. ``seq_lens``
count every context token including this step's new ones.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BF16_NAN = np.uint16(0x7FC0)
POOL_CHUNK = 1 << 24


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    n = int(np.prod(shape))
    return to_bf16_bits(rng.standard_normal(n, dtype=np.float32)).reshape(shape)


@dataclass
class Workload:
    """One batch of a paged-attention step, as numpy arrays (bf16 as uint16)."""

    name: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    seq_lens: np.ndarray      # int32 [B]
    query_lens: np.ndarray    # int32 [B]
    cu_seqlens: np.ndarray    # int32 [B+1]
    block_table: np.ndarray   # int32 [B, max_blocks], -1 beyond each request's blocks
    slot_mapping: np.ndarray  # int32 [T]
    q: np.ndarray             # uint16 [T, H, D]
    k_new: np.ndarray         # uint16 [T, Hkv, D]
    v_new: np.ndarray         # uint16 [T, Hkv, D]
    pool: np.ndarray          # uint16 [2, NB, BS, Hkv, D], before this step's write
    seed: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def max_query_len(self) -> int:
        return int(self.query_lens.max()) if self.num_seqs else 0

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.num_seqs else 0

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def kv_bytes_per_token(self) -> int:
        """K and V bytes of one token of one layer (bf16)."""
        return 2 * self.num_kv_heads * self.head_dim * 2

    def kv_bytes(self, decode_only: bool = False) -> int:
        """Algorithmic KV bytes: every request reads its whole context once."""
        lens = self.seq_lens if not decode_only else self.seq_lens[self.query_lens == 1]
        return int(lens.astype(np.int64).sum()) * self.kv_bytes_per_token

    def unique_kv_bytes(self) -> int:
        """KV bytes counting each physical slot once (shared prefixes once)."""
        slots = set()
        for i in range(self.num_seqs):
            n = int(self.seq_lens[i])
            nblk = -(-n // self.block_size)
            for b in range(nblk):
                used = min(self.block_size, n - b * self.block_size)
                slots.add((int(self.block_table[i, b]), used))
        per_block: dict[int, int] = {}
        for blk, used in slots:
            per_block[blk] = max(per_block.get(blk, 0), used)
        return sum(per_block.values()) * self.kv_bytes_per_token

    def attention_flops(self, min_query_len: int = 1) -> int:
        """Causal-exact attention FLOPs (QK^T and PV) of requests with q >= min_query_len."""
        total = 0
        for i in range(self.num_seqs):
            ql = int(self.query_lens[i])
            if ql < min_query_len:
                continue
            L = int(self.seq_lens[i])
            # query j sees pos_j + 1 = L - ql + j + 1 keys
            keys = ql * (L - ql) + ql * (ql + 1) // 2
            total += 4 * self.head_dim * keys * self.num_heads
        return total


def build(name: str, seq_lens, query_lens, num_heads: int, num_kv_heads: int, head_dim: int,
          block_size: int = 16, seed: int = 0, rng: np.random.Generator | None = None,
          pool_factor: float = 1.25, num_blocks: int | None = None,
          shared_prefix: list[tuple[list[int], int]] | None = None,
          max_blocks: int | None = None, poison: bool = True, scale: float | None = None,
          meta: dict | None = None) -> Workload:
    """Build a workload from explicit lengths.

    ``shared_prefix`` lists groups as ``(request indices, prefix tokens)``;
    the prefix (a whole number of blocks) is allocated once per group and its
    physical blocks appear in every member's block table (copy-on-write
    sharing of page 2's PagedAttention deep-dive). The draws happen in this
    order: block permutation, q, k_new, v_new, then the pool from a child
    generator.
    """
    if rng is None:
        rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    query_lens = np.asarray(query_lens, dtype=np.int64)
    B = int(seq_lens.shape[0])
    assert query_lens.shape == (B,)
    assert np.all(query_lens >= 0) and np.all(seq_lens >= query_lens)
    BS = block_size
    nblk = -(-seq_lens // BS)

    shared_of: dict[int, tuple[int, int]] = {}
    if shared_prefix:
        for g, (members, ptoks) in enumerate(shared_prefix):
            assert ptoks % BS == 0
            for m in members:
                assert seq_lens[m] - query_lens[m] >= ptoks, "prefix must be cached history"
                shared_of[int(m)] = (g, ptoks // BS)
    need = int(nblk.sum())
    if shared_prefix:
        for g, (members, ptoks) in enumerate(shared_prefix):
            need -= (len(members) - 1) * (ptoks // BS)
    if num_blocks is None:
        num_blocks = max(1, math.ceil(pool_factor * need))
    assert num_blocks >= need, "pool too small for the requested lengths"
    if max_blocks is None:
        max_blocks = max(1, int(nblk.max()) if B else 1)

    perm = rng.permutation(num_blocks).astype(np.int32)
    cursor = 0
    group_blocks: dict[int, np.ndarray] = {}
    table = np.full((max(B, 0), max_blocks), -1, dtype=np.int32)
    for i in range(B):
        start = 0
        if i in shared_of:
            g, pblocks = shared_of[i]
            if g not in group_blocks:
                group_blocks[g] = perm[cursor:cursor + pblocks]
                cursor += pblocks
            table[i, :pblocks] = group_blocks[g]
            start = pblocks
        n = int(nblk[i]) - start
        table[i, start:start + n] = perm[cursor:cursor + n]
        cursor += n

    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(query_lens)
    T = int(cu[-1])
    H, Hkv, D = num_heads, num_kv_heads, head_dim

    slot_mapping = np.empty(T, dtype=np.int32)
    history = np.zeros(num_blocks * BS, dtype=bool)
    for i in range(B):
        L, ql = int(seq_lens[i]), int(query_lens[i])
        pos = np.arange(L, dtype=np.int64)
        slots = table[i, pos // BS].astype(np.int64) * BS + pos % BS
        history[slots[:L - ql]] = True
        slot_mapping[cu[i]:cu[i + 1]] = slots[L - ql:]

    q = _normal_bf16(rng, (T, H, D))
    k_new = _normal_bf16(rng, (T, Hkv, D))
    v_new = _normal_bf16(rng, (T, Hkv, D))

    pool_rng = np.random.default_rng(rng.integers(0, 2**63 - 1))
    pool = np.empty((2, num_blocks, BS, Hkv, D), dtype=np.uint16)
    flat = pool.reshape(-1)
    for start in range(0, flat.shape[0], POOL_CHUNK):
        stop = min(flat.shape[0], start + POOL_CHUNK)
        flat[start:stop] = to_bf16_bits(pool_rng.standard_normal(stop - start, dtype=np.float32))
    by_slot = pool.reshape(2, num_blocks * BS, Hkv * D)
    by_slot[:, ~history, :] = BF16_NAN if poison else np.uint16(0)

    return Workload(
        name=name, num_heads=H, num_kv_heads=Hkv, head_dim=D, block_size=BS,
        num_blocks=int(num_blocks), scale=(1.0 / math.sqrt(D)) if scale is None else scale,
        seq_lens=seq_lens.astype(np.int32), query_lens=query_lens.astype(np.int32),
        cu_seqlens=cu, block_table=table, slot_mapping=slot_mapping, q=q, k_new=k_new,
        v_new=v_new, pool=pool, seed=seed, meta=dict(meta or {}))


# ----------------------------------------------------------------------------
# The five workloads of the method's hot path (one attention layer each).
# ----------------------------------------------------------------------------

def tiny(seed: int = 1, poison: bool = True) -> Workload:
    """4 decode requests with contexts {1,7,16,33}; 4 q / 2 kv heads, D 64,
    block 16, a 64-block pool whose tables take blocks from a seeded
    permutation, scale 1/8; the 4 new K/V rows are written via slot_mapping."""
    return build("tiny", [1, 7, 16, 33], [1, 1, 1, 1], 4, 2, 64, 16, seed=seed,
                 num_blocks=64, max_blocks=3, poison=poison, scale=1.0 / 8.0)


def llama_decode(seed: int = 2, poison: bool = True, batch: int = 64) -> Workload:
    """Llama-3-8B decode shape: batch 64, q 1, contexts U[512,4096], 32/8 heads,
    D 128, block 16, pool 1.25x the need."""
    rng = np.random.default_rng(seed)
    L = rng.integers(512, 4096, size=batch, endpoint=True)
    return build("llama3_8b_decode", L, np.ones(batch, dtype=np.int64), 32, 8, 128, 16,
                 seed=seed, rng=rng, max_blocks=4096 // 16, poison=poison)


def long_decode(seed: int = 3, poison: bool = True, batch: int = 8,
                lo: int = 32768, hi: int = 131072) -> Workload:
    """Long-context decode: batch 8, contexts U[32768,131072], 32/8, D 128,
    split into 512-token partitions merged by log-sum-exp."""
    rng = np.random.default_rng(seed)
    L = rng.integers(lo, hi, size=batch, endpoint=True)
    return build("long_split_kv", L, np.ones(batch, dtype=np.int64), 32, 8, 128, 16, seed=seed,
                 rng=rng, max_blocks=-(-hi // 16), poison=poison,
                 meta={"partition_size": 512})


def prefix_shared(seed: int = 4, poison: bool = True, groups: int = 4, per_group: int = 64,
                  prefix_tokens: int = 2048, tail_lo: int = 64, tail_hi: int = 1024) -> Workload:
    """Copy-on-write prefix sharing: 4 groups x 64 decode requests; each group
    shares one 2048-token prefix (whole blocks) and has private tails of
    U[64,1024] tokens; 32/8, D 128."""
    rng = np.random.default_rng(seed)
    B = groups * per_group
    tails = rng.integers(tail_lo, tail_hi, size=B, endpoint=True)
    L = prefix_tokens + tails
    sp = [(list(range(g * per_group, (g + 1) * per_group)), prefix_tokens) for g in range(groups)]
    return build("prefix_cow", L, np.ones(B, dtype=np.int64), 32, 8, 128, 16, seed=seed, rng=rng,
                 shared_prefix=sp, max_blocks=-(-(prefix_tokens + tail_hi) // 16), poison=poison,
                 meta={"groups": groups, "per_group": per_group,
                       "prefix_tokens": prefix_tokens})


def mixed_step(seed: int = 5, poison: bool = True, decodes: int = 48, chunks: int = 4,
               chunk_len: int = 512, budget: int = 8192) -> Workload:
    """Mixed continuous-batching step: 48 decodes (contexts U[256,8192]) then
    4 prefill chunks of 512 queries over a prior context U[0,8192]; causal;
    token budget 8192; every new K/V written via slot_mapping; 32/8, D 128."""
    rng = np.random.default_rng(seed)
    Ld = rng.integers(256, 8192, size=decodes, endpoint=True)
    prior = rng.integers(0, 8192, size=chunks, endpoint=True)
    L = np.concatenate([Ld, prior + chunk_len])
    ql = np.concatenate([np.ones(decodes, dtype=np.int64), np.full(chunks, chunk_len)])
    assert int(ql.sum()) <= budget
    return build("mixed_step", L, ql, 32, 8, 128, 16, seed=seed, rng=rng,
                 max_blocks=-(-(8192 + chunk_len) // 16), poison=poison,
                 meta={"token_budget": budget})


def prefill_chunks(seed: int = 5, poison: bool = True, chunks: int = 4,
                   chunk_len: int = 512) -> Workload:
    """The prefill part of the mixed step on its own: the same 4 chunks of 512
    queries over the same prior contexts (drawn exactly as mixed_step draws
    them, after its 48 decode lengths); causal; 32/8, D 128."""
    rng = np.random.default_rng(seed)
    rng.integers(256, 8192, size=48, endpoint=True)  # mixed_step's decode lengths
    prior = rng.integers(0, 8192, size=chunks, endpoint=True)
    L = prior + chunk_len
    ql = np.full(chunks, chunk_len)
    return build("prefill_chunks", L, ql, 32, 8, 128, 16, seed=seed, rng=rng,
                 max_blocks=-(-(8192 + chunk_len) // 16), poison=poison)


def spec_verify(seed: int = 6, poison: bool = True, batch: int = 64, lo_q: int = 2,
                hi_q: int = 8) -> Workload:
    """Speculative-decoding verification step on the Llama-3-8B decode shape:
    batch 64, each request verifies q ~ U[2, 8] drafted tokens (causal among
    them) over a context U[512, 4096] that includes them; 32/8, D 128."""
    rng = np.random.default_rng(seed)
    L = rng.integers(512, 4096, size=batch, endpoint=True)
    ql = rng.integers(lo_q, hi_q, size=batch, endpoint=True)
    return build("spec_verify", L, ql, 32, 8, 128, 16, seed=seed, rng=rng,
                 max_blocks=4096 // 16, poison=poison)


CONFIGS = {
    "tiny": tiny,
    "llama3_8b_decode": llama_decode,
    "long_split_kv": long_decode,
    "prefix_cow": prefix_shared,
    "mixed_step": mixed_step,
    "prefill_chunks": prefill_chunks,
    "spec_verify": spec_verify,
}


def cascade_inputs(w: Workload, groups) -> dict:
    """Inputs of the shared-prefix (cascade) call for a workload whose
    requests share copy-on-write prefixes: ``groups`` lists (first request,
    count, prefix tokens), contiguous and in order; requests after the last
    group have no prefix. Returns the group starts, prefix lengths and
    tables, and every request's tail table (its blocks after the prefix) and
    tail length, as int32 numpy arrays, plus the maxima the call takes."""
    bs = w.block_size
    starts = [0]
    for first, count, _ in groups:
        assert first == starts[-1], "groups must be contiguous and start at request 0"
        starts.append(first + count)
    prefix_of = np.zeros(w.num_seqs, dtype=np.int64)
    for first, count, ptok in groups:
        assert ptok % bs == 0
        prefix_of[first:first + count] = ptok
    max_pb = max([p // bs for _, _, p in groups] + [1])
    ptables = np.full((max(len(groups), 1), max_pb), -1, dtype=np.int32)
    for gi, (first, count, ptok) in enumerate(groups):
        ptables[gi, :ptok // bs] = w.block_table[first, :ptok // bs]
        assert (w.block_table[first:first + count, :ptok // bs] == ptables[gi, :ptok // bs]).all()
    tail_lens = (w.seq_lens - prefix_of).astype(np.int32)
    ttables = np.full((w.num_seqs, w.max_blocks), -1, dtype=np.int32)
    for i in range(w.num_seqs):
        nb_i = -(-int(tail_lens[i]) // bs)
        off = int(prefix_of[i]) // bs
        ttables[i, :nb_i] = w.block_table[i, off:off + nb_i]
    return {
        "group_starts": np.array(starts, dtype=np.int32),
        "prefix_lens": np.array([p for _, _, p in groups] or [0], dtype=np.int32)[:len(groups)],
        "prefix_tables": ptables[:len(groups)] if groups else ptables[:0],
        "max_group_size": max([c for _, c, _ in groups] + [1]),
        "max_prefix_len": max([p for _, _, p in groups] + [0]),
        "tail_tables": ttables,
        "tail_lens": tail_lens,
        "max_tail_len": int(tail_lens.max()),
    }


def prefix_groups(w: Workload) -> list:
    """The (first request, count, prefix tokens) groups of a prefix_shared workload."""
    pg, g, ptok = w.meta["per_group"], w.meta["groups"], w.meta["prefix_tokens"]
    return [(k * pg, pg, ptok) for k in range(g)]


def permute_requests(w: Workload, order) -> Workload:
    """The same requests in another order (cu_seqlens, tables and tokens
    follow); the pool is unchanged."""
    order = np.asarray(order, dtype=np.int64)
    ql = w.query_lens[order]
    cu = np.zeros(len(order) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(ql)
    tok = np.concatenate([np.arange(w.cu_seqlens[i], w.cu_seqlens[i + 1]) for i in order]) \
        if len(order) else np.zeros(0, dtype=np.int64)
    return Workload(
        name=w.name + "_permuted", num_heads=w.num_heads, num_kv_heads=w.num_kv_heads,
        head_dim=w.head_dim, block_size=w.block_size, num_blocks=w.num_blocks, scale=w.scale,
        seq_lens=w.seq_lens[order].copy(), query_lens=ql.copy(), cu_seqlens=cu,
        block_table=w.block_table[order].copy(), slot_mapping=w.slot_mapping[tok].copy(),
        q=w.q[tok].copy(), k_new=w.k_new[tok].copy(), v_new=w.v_new[tok].copy(),
        pool=w.pool, seed=w.seed, meta=dict(w.meta, order=order.tolist()))
