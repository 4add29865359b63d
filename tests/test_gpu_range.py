"""Attention over key ranges and sequence-parallel merging (needs a GB300).

Page 1 (从 token 调度到采样输出…), §07: sequence parallelism splits the
sequence dimension and renormalises the pieces with log-sum-exp. The range
call's piece for keys [s, e) of a request must equal the oracle's attention
restricted to those keys (every row, within 2e-3; rows that see no key of
the range give out 0 and lse -inf), and the pieces of a context cut into
ranks' ranges, merged by pkv_lse_merge, must equal the oracle over the whole
context. The last test runs two real processes on the one GPU that exchange
their pieces over gloo.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from paged_kv_cache_varlen_gb300 import binding as pkv
from paged_kv_cache_varlen_gb300 import seqpar
from paged_kv_cache_varlen_gb300 import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _batch(head_dim=128):
    # decodes (one split into partitions), a verification step, two prefill
    # chunks (one with no prior context), 32/8 heads, D 128 (or 64)
    return wl.build("range", [6000, 700, 1800, 520, 2400], [1, 1, 300, 5, 512], 32, 8, head_dim,
                    seed=41)


def _range_call(dev, w, ranges, partition_size=-1):
    """One range call over per-request key ranges (s_i, e_i); returns the
    pieces for every token."""
    keep = [i for i, (s, e) in enumerate(ranges) if e > s]
    tables, lens, ks, qs = [], [], [], []
    for i in keep:
        s, e = ranges[i]
        nb = -(-(e - s) // w.block_size)
        tables.append(w.block_table[i, s // w.block_size:s // w.block_size + nb])
        lens.append(e - s)
        ks.append(s)
        qs.append(int(w.seq_lens[i] - w.query_lens[i]))
    width = max(len(t) for t in tables)
    table = np.full((len(keep), width), -1, dtype=np.int32)
    for r, t in enumerate(tables):
        table[r, :len(t)] = t
    tok, cu = seqpar.compact_queries(w.cu_seqlens, np.array(keep))
    tok_t = torch.from_numpy(tok).cuda()
    q = dev.q.index_select(0, tok_t).contiguous()
    out = torch.full((len(tok), w.num_heads, w.head_dim), float("nan"), device="cuda")
    lse = torch.full((len(tok), w.num_heads), float("nan"), device="cuda")
    pkv.paged_attention_varlen_range(
        q, dev.pool, gu.i32_tensor(table), gu.i32_tensor(cu), gu.i32_tensor(np.array(lens)),
        gu.i32_tensor(np.array(ks)), gu.i32_tensor(np.array(qs)),
        int(w.query_lens[keep].max()), int(max(lens)), out=out, out_lse=lse, scale=w.scale,
        partition_size=partition_size, dev_status=dev.status)
    assert dev.dev_status() == 0
    return tok, out, lse


def _oracle_pieces(oracle, w, ref_pool, ranges, tok):
    ref_o = np.zeros((len(tok), w.num_heads, w.head_dim))
    ref_l = np.zeros((len(tok), w.num_heads))
    pos = {int(t): k for k, t in enumerate(tok)}
    for i, (s, e) in enumerate(ranges):
        if e <= s:
            continue
        rows = np.arange(w.cu_seqlens[i], w.cu_seqlens[i + 1], dtype=np.int32)
        o, ls = oracle.paged_attention(w.q, ref_pool, w.block_table, w.cu_seqlens, w.seq_lens,
                                       w.scale, rows=rows, key_begin=s, key_end=e)
        idx = [pos[int(r)] for r in rows]
        ref_o[idx], ref_l[idx] = o, ls
    return ref_o, ref_l


def _compare_pieces(out, lse, ref_o, ref_l):
    o = out.cpu().numpy().astype(np.float64)
    ls = lse.cpu().numpy().astype(np.float64)
    empty = np.isneginf(ref_l)
    assert np.array_equal(np.isneginf(ls), empty), "rows with no visible key differ"
    assert np.all(o[empty] == 0.0)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(ls[~empty]))
    err_o = float(np.abs(o - ref_o).max())
    err_l = float(np.abs(ls[~empty] - ref_l[~empty]).max()) if (~empty).any() else 0.0
    assert err_o <= gu.ATOL and err_l <= gu.ATOL, (err_o, err_l)


@pytest.mark.parametrize("case", ["head", "tail", "middle", "past_the_queries", "whole"])
def test_range_piece_matches_oracle(oracle, case):
    _check_case(oracle, case, 128)


@pytest.mark.parametrize("case", ["middle", "past_the_queries", "whole"])
def test_range_piece_head_dim_64(oracle, case):
    _check_case(oracle, case, 64)


def _check_case(oracle, case, head_dim):
    w = _batch(head_dim)
    ref_pool = oracle.kv_cache_write(w.pool, w.k_new, w.v_new, w.slot_mapping)
    dev = gu.DeviceStep(w)
    dev.write()
    ranges = []
    for L, q in zip(w.seq_lens.tolist(), w.query_lens.tolist()):
        half = (L // 2) // 16 * 16
        if case == "head":
            ranges.append((0, max(16, half)))
        elif case == "tail":
            ranges.append((half, L))
        elif case == "middle":
            ranges.append((min(L - 1, 256) // 16 * 16, max(L - q - 16, 272)))
        elif case == "past_the_queries":
            # keys from just before the first query: early queries of a chunk see
            # only part of it, and a range starting after every query is empty
            ranges.append(((L - q) // 16 * 16, L))
        else:
            ranges.append((0, L))
    ranges = [(s, min(e, int(L))) for (s, e), L in zip(ranges, w.seq_lens)]
    tok, out, lse = _range_call(dev, w, ranges)
    ref_o, ref_l = _oracle_pieces(oracle, w, ref_pool, ranges, tok)
    _compare_pieces(out, lse, ref_o, ref_l)
    if case == "whole":   # the whole range is the ordinary call, bit for bit
        full, full_lse = dev.attend()
        tok_t = torch.from_numpy(tok).cuda()
        assert torch.equal(full[tok_t], out) and torch.equal(full_lse[tok_t], lse)


def test_range_with_no_visible_key():
    """A range that starts after every query of a request: all its rows are
    empty pieces (out 0, lse -inf)."""
    w = wl.build("range_empty", [600], [40], 32, 8, 128, seed=43)
    dev = gu.DeviceStep(w)
    dev.write()
    tables = w.block_table[:, 0:38]
    lens = np.array([600], dtype=np.int32)
    out = torch.full((40, 32, 128), float("nan"), device="cuda")
    lse = torch.full((40, 32), float("nan"), device="cuda")
    pkv.paged_attention_varlen_range(
        dev.q, dev.pool, gu.i32_tensor(tables), dev.cu, gu.i32_tensor(lens),
        gu.i32_tensor(np.array([1000])), gu.i32_tensor(np.array([560])), 40, 600, out=out,
        out_lse=lse, scale=w.scale, dev_status=dev.status)
    assert dev.dev_status() == 0
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


@pytest.mark.parametrize("world", [2, 3])
def test_sequence_parallel_pieces_merge_to_full_attention(oracle, world):
    w = _batch()
    ref_pool = oracle.kv_cache_write(w.pool, w.k_new, w.v_new, w.slot_mapping)
    dev = gu.DeviceStep(w)
    dev.write()
    pieces = [seqpar.rank_piece(dev.q, dev.pool, w.block_table, w.cu_seqlens, w.seq_lens, r,
                                world, w.scale, dev_status=dev.status) for r in range(world)]
    assert dev.dev_status() == 0
    po = torch.stack([p[0] for p in pieces]).contiguous()
    pl = torch.stack([p[1] for p in pieces]).contiguous()
    out, lse = seqpar.merge_pieces(po, pl)
    ref_o, ref_l = oracle.paged_attention(w.q, ref_pool, w.block_table, w.cu_seqlens, w.seq_lens,
                                          w.scale)
    gu.compare(out, lse, ref_o, ref_l)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import oracle
    from paged_kv_cache_varlen_gb300 import seqpar as sp
    from tests import gpu_util as g

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        torch.cuda.set_device(0)
        w = _batch()
        dev = g.DeviceStep(w)   # every process holds the same seeded pool
        dev.write()
        o, ls = sp.rank_piece(dev.q, dev.pool, w.block_table, w.cu_seqlens, w.seq_lens, rank,
                              world, w.scale, dev_status=dev.status)
        status = dev.dev_status()
        po, pl = sp.gather_pieces(o, ls)
        out, lse = sp.merge_pieces(po, pl)
        torch.cuda.synchronize()
        if rank == 0:
            orc = oracle.load()
            ref_pool = orc.kv_cache_write(w.pool, w.k_new, w.v_new, w.slot_mapping)
            ref_o, ref_l = orc.paged_attention(w.q, ref_pool, w.block_table, w.cu_seqlens,
                                               w.seq_lens, w.scale)
            err_o = float(np.abs(out.cpu().numpy() - ref_o).max())
            err_l = float(np.abs(lse.cpu().numpy() - ref_l).max())
            np.save(os.path.join(out_dir, "result.npy"), np.array([err_o, err_l, status]))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_processes_exchange_pieces_over_gloo(tmp_path):
    """Two processes, each attending to its key range on the one GPU (they
    never wait on each other inside a kernel), exchange their pieces over a
    gloo group and merge them with pkv_lse_merge."""
    mp.start_processes(_rank_main, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    err_o, err_l, status = np.load(tmp_path / "result.npy")
    assert status == 0
    assert err_o <= gu.ATOL and err_l <= gu.ATOL
