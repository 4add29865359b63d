"""Sequence-parallel sharding on the host (CPU only, no GPU).

Page 1 (从 token 调度到采样输出…), §07: sequence parallelism splits the
prompt dimension and renormalises the pieces with log-sum-exp. Here the
bookkeeping of ``seqpar`` is checked: the key ranges cover each context
exactly once at block boundaries, a rank's shifted block table names the
same physical slots as the whole table, and its positions reproduce the
causal limits. Then two gloo ranks exchange pieces the oracle computed over
their ranges and the merged result equals the oracle on the whole context.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from paged_kv_cache_varlen_gb300 import seqpar  # noqa: E402
from paged_kv_cache_varlen_gb300 import workloads as wl  # noqa: E402


@pytest.mark.parametrize("L,world", [(1, 2), (16, 2), (17, 2), (1000, 3), (4096, 4), (33, 8)])
def test_key_ranges_cover_the_context_once(L, world):
    r = seqpar.key_ranges(L, world, 16)
    assert len(r) == world
    assert r[0][0] == 0 and r[-1][1] == L
    for (s0, e0), (s1, e1) in zip(r, r[1:]):
        assert e0 == s1                  # contiguous, no overlap
    for s, e in r:
        assert s <= e
        assert s % 16 == 0 or s == e == L  # block-aligned starts; empty ranges at the end
    sizes = [-(-(e - s) // 16) for s, e in r]
    assert max(sizes) - min(sizes) <= 1  # as even as whole blocks allow


def test_shard_inputs_name_the_same_slots():
    w = wl.build("sp", [5000, 40, 1800, 3], [1, 1, 300, 2], 32, 8, 128, seed=5)
    for world in (2, 3):
        covered = [np.zeros(int(L), dtype=int) for L in w.seq_lens]
        for rank in range(world):
            sh = seqpar.shard_inputs(w.block_table, w.seq_lens, w.query_lens, rank, world, 16)
            for r, i in enumerate(sh["keep"]):
                s = int(sh["key_start_pos"][r])
                n = int(sh["seq_lens"][r])
                p = np.arange(n)
                local = sh["block_table"][r, p // 16] * 16 + p % 16
                glob = w.block_table[i, (s + p) // 16] * 16 + (s + p) % 16
                assert np.array_equal(local, glob)
                covered[i][s:s + n] += 1
                # query j sits at L - q + j, as in the ordinary call
                assert sh["query_start_pos"][r] == w.seq_lens[i] - w.query_lens[i]
        for c in covered:
            assert np.all(c == 1)        # every key in exactly one rank's range


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


WORLD = 2


def _rank_main(rank, port, out_dir):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import oracle
    from paged_kv_cache_varlen_gb300 import seqpar as sp
    from paged_kv_cache_varlen_gb300 import workloads as w_

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        orc = oracle.load()
        w = w_.build("sp", [700, 90, 400], [1, 1, 40], 8, 2, 64, seed=9)
        pool = orc.kv_cache_write(w.pool, w.k_new, w.v_new, w.slot_mapping)
        T, H, D = w.q.shape
        out = np.zeros((T, H, D))
        lse = np.full((T, H), -np.inf)
        for i in range(w.num_seqs):   # the oracle stands in for this rank's device call
            s, e = sp.key_ranges(int(w.seq_lens[i]), WORLD, 16)[rank]
            rows = np.arange(w.cu_seqlens[i], w.cu_seqlens[i + 1], dtype=np.int32)
            o, ls = orc.paged_attention(w.q, pool, w.block_table, w.cu_seqlens, w.seq_lens,
                                        w.scale, rows=rows, key_begin=s, key_end=e)
            out[rows], lse[rows] = o, ls
        po, pl = sp.gather_pieces(torch.from_numpy(out), torch.from_numpy(lse))
        mo, ml = orc.lse_merge(po.numpy(), pl.numpy())
        ref_o, ref_l = orc.paged_attention(w.q, pool, w.block_table, w.cu_seqlens, w.seq_lens,
                                           w.scale)
        np.save(os.path.join(out_dir, f"err{rank}.npy"),
                np.array([np.abs(mo - ref_o).max(), np.abs(ml - ref_l).max(), po.shape[0]]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_merge_to_the_whole_context(tmp_path):
    mp.start_processes(_rank_main, args=(_free_port(), str(tmp_path)), nprocs=WORLD, join=True,
                       start_method="spawn")
    for r in range(WORLD):
        err_o, err_l, parts = np.load(tmp_path / f"err{r}.npy")
        assert parts == WORLD
        assert err_o < 1e-12 and err_l < 1e-12
