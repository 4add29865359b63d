"""Guard bands around every buffer the kernels write (needs a GB300).

The memory checker is not available on this GPU pool, so out-of-bounds
stores are caught this way instead: each output, workspace and pool sits
inside a larger buffer whose bands before and after hold a sentinel bit
pattern, and after the call the bands must be unchanged. The calls cover
every kernel that writes device memory -- KV write, block copies, decode,
split-KV merge, prefill, the public merge, the cascade call, the key-range
call and the allocation-free call -- on shapes with ragged tails (partial
blocks, partial 128-row tiles, partial partitions). Outputs start as NaN
(the sentinel), so rows never written also fail the parity check.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_varlen_gb300 import binding as pkv
from paged_kv_cache_varlen_gb300 import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
G = 8192  # guard elements on each side


def _mixed(head_dim, num_heads=32, num_kv_heads=8):
    # decodes (one split into many partitions), verification steps (5 and 8
    # queries), prefill chunks with ragged tiles (300 and 513 queries)
    return wl.build("guards", [3001, 17, 1, 900, 2050, 1300, 4000],
                    [1, 1, 1, 5, 300, 8, 513], num_heads, num_kv_heads, head_dim, seed=91)


def _device_inputs(w):
    q = gu.bf16_tensor(w.q)
    return (q, gu.i32_tensor(w.block_table), gu.i32_tensor(w.cu_seqlens),
            gu.i32_tensor(w.seq_lens))


@pytest.mark.parametrize("head_dim", [128, 64])
def test_kv_write_stays_inside_the_pool(oracle, head_dim):
    w = _mixed(head_dim)
    ref = oracle.kv_cache_write(w.pool, w.k_new, w.v_new, w.slot_mapping)
    buf, pool = gu.guarded(w.pool.shape, torch.bfloat16, G)
    pool.copy_(gu.bf16_tensor(w.pool))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.kv_cache_write(pool, gu.bf16_tensor(w.k_new), gu.bf16_tensor(w.v_new),
                       gu.i32_tensor(w.slot_mapping), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert gu.guards_intact(buf, pool.numel(), G)
    assert torch.equal(pool.view(torch.int16), gu.bf16_tensor(ref).view(torch.int16))


@pytest.mark.parametrize("head_dim,partition_size", [(128, 256), (128, -1), (64, 128)])
def test_attention_stays_inside_its_buffers(oracle, head_dim, partition_size):
    w = _mixed(head_dim)
    ref_pool = oracle.kv_cache_write(w.pool, w.k_new, w.v_new, w.slot_mapping)
    pool = gu.bf16_tensor(ref_pool)
    q, table, cu, lens = _device_inputs(w)
    T, H, D = w.q.shape
    ob, out = gu.guarded((T, H, D), torch.float32, G)
    lb, lse = gu.guarded((T, H), torch.float32, G)
    need = pkv.attention_workspace_size(w.num_seqs, T, H, w.num_kv_heads, D, w.max_seq_len,
                                        partition_size)
    wb, ws = gu.guarded((need,), torch.uint8, G)
    ws.zero_()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):  # a second call reuses the workspace the first left behind
        pkv.paged_attention_varlen(q, pool, table, cu, lens, w.max_query_len, w.max_seq_len,
                                   out=out, out_lse=lse, scale=w.scale,
                                   partition_size=partition_size, workspace=ws,
                                   dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert gu.guards_intact(ob, out.numel(), G), "store outside out"
    assert gu.guards_intact(lb, lse.numel(), G), "store outside out_lse"
    assert gu.guards_intact(wb, ws.numel(), G), "store outside the workspace"
    # the work tickets are zero again at the end of the workspace
    assert int(ws[-256:].count_nonzero()) == 0
    ref_o, ref_l = oracle.paged_attention(w.q, ref_pool, w.block_table, w.cu_seqlens, w.seq_lens,
                                          w.scale)
    gu.compare(out, lse, ref_o, ref_l)


def test_public_merge_stays_inside_its_buffers(oracle):
    rng = np.random.default_rng(5)
    P, T, H, D = 7, 33, 8, 128
    po = rng.standard_normal((P, T, H, D)).astype(np.float32)
    pl = rng.standard_normal((P, T, H)).astype(np.float32) * 3
    pl[2] = -np.inf
    ob, out = gu.guarded((T, H, D), torch.float32, G)
    lb, lse = gu.guarded((T, H), torch.float32, G)
    pkv.lse_merge(torch.from_numpy(po).cuda(), torch.from_numpy(pl).cuda(), out=out, out_lse=lse)
    torch.cuda.synchronize()
    assert gu.guards_intact(ob, out.numel(), G) and gu.guards_intact(lb, lse.numel(), G)
    ref_o, ref_l = oracle.lse_merge(po.astype(np.float64), pl.astype(np.float64))
    assert np.abs(out.cpu().numpy() - ref_o).max() <= 1e-4
    assert np.abs(lse.cpu().numpy() - ref_l).max() <= 1e-4


def test_copy_blocks_stays_inside_the_pool():
    w = _mixed(128)
    buf, pool = gu.guarded(w.pool.shape, torch.bfloat16, G)
    pool.copy_(gu.bf16_tensor(w.pool))
    before = pool.clone()
    src = torch.tensor([0, 5, w.num_blocks - 1], dtype=torch.int32, device="cuda")
    dst = torch.tensor([3, 9, 7], dtype=torch.int32, device="cuda")
    pkv.copy_blocks(pool, src, dst)
    torch.cuda.synchronize()
    assert gu.guards_intact(buf, pool.numel(), G)
    for s_, d_ in zip(src.tolist(), dst.tolist()):
        assert torch.equal(pool[:, d_].view(torch.int16), before[:, s_].view(torch.int16))


def test_cascade_stays_inside_its_buffers(oracle):
    sizes, prefixes = [3, 70, 2], [48, 512, 0]
    rng = np.random.default_rng(93)
    lens, sp, groups, first = [], [], [], 0
    for n, ptok in zip(sizes, prefixes):
        tails = rng.integers(1, 300, size=n, endpoint=True)
        lens += (ptok + tails).tolist()
        if ptok:
            sp.append((list(range(first, first + n)), ptok))
        groups.append((first, n, ptok))
        first += n
    w = wl.build("guards_cascade", lens, [1] * len(lens), 32, 8, 128, seed=94, shared_prefix=sp)
    ref_pool = oracle.kv_cache_write(w.pool, w.k_new, w.v_new, w.slot_mapping)
    pool = gu.bf16_tensor(ref_pool)
    ci = wl.cascade_inputs(w, groups)
    B, H, D = w.q.shape
    ob, out = gu.guarded((B, H, D), torch.float32, G)
    lb, lse = gu.guarded((B, H), torch.float32, G)
    need = pkv.cascade_workspace_size(B, len(ci["prefix_lens"]), ci["max_group_size"],
                                      ci["max_prefix_len"], ci["max_tail_len"], H, 8, D)
    wb, ws = gu.guarded((need,), torch.uint8, G)
    ws.zero_()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.cascade_decode(gu.bf16_tensor(w.q), pool, gu.i32_tensor(ci["group_starts"]),
                       gu.i32_tensor(ci["prefix_lens"]), gu.i32_tensor(ci["prefix_tables"]),
                       ci["max_group_size"], ci["max_prefix_len"],
                       gu.i32_tensor(ci["tail_tables"]), gu.i32_tensor(ci["tail_lens"]),
                       ci["max_tail_len"], out=out, out_lse=lse, scale=w.scale, workspace=ws,
                       dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert gu.guards_intact(ob, out.numel(), G) and gu.guards_intact(lb, lse.numel(), G)
    assert gu.guards_intact(wb, ws.numel(), G)
    ref_o, ref_l = oracle.paged_attention(w.q, ref_pool, w.block_table, w.cu_seqlens, w.seq_lens,
                                          w.scale)
    gu.compare(out, lse, ref_o, ref_l)


def test_range_and_noalloc_calls_stay_inside_their_buffers(oracle):
    w = _mixed(128)
    ref_pool = oracle.kv_cache_write(w.pool, w.k_new, w.v_new, w.slot_mapping)
    pool = gu.bf16_tensor(ref_pool)
    q, table, cu, lens = _device_inputs(w)
    T, H, D = w.q.shape
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # the second half of every context as the key range
    ks = (w.seq_lens // 2) // 16 * 16
    tab = np.full_like(w.block_table, -1)
    for i, s in enumerate(ks):
        nb = -(-(int(w.seq_lens[i]) - int(s)) // 16)
        tab[i, :nb] = w.block_table[i, s // 16:s // 16 + nb]
    ob, out = gu.guarded((T, H, D), torch.float32, G)
    lb, lse = gu.guarded((T, H), torch.float32, G)
    rl = (w.seq_lens - ks).astype(np.int32)
    need = pkv.attention_workspace_size(w.num_seqs, T, H, 8, D, int(rl.max()), 256)
    wb, ws = gu.guarded((need,), torch.uint8, G)
    ws.zero_()
    pkv.paged_attention_varlen_range(
        q, pool, gu.i32_tensor(tab), cu, gu.i32_tensor(rl), gu.i32_tensor(ks),
        gu.i32_tensor(w.seq_lens - w.query_lens), w.max_query_len, int(rl.max()), out=out,
        out_lse=lse, scale=w.scale, partition_size=256, workspace=ws, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert gu.guards_intact(ob, out.numel(), G) and gu.guards_intact(lb, lse.numel(), G)
    assert gu.guards_intact(wb, ws.numel(), G)
    for i in range(w.num_seqs):
        rows = np.arange(w.cu_seqlens[i], w.cu_seqlens[i + 1], dtype=np.int32)
        ro, rlse = oracle.paged_attention(w.q, ref_pool, w.block_table, w.cu_seqlens, w.seq_lens,
                                          w.scale, rows=rows, key_begin=int(ks[i]))
        got_o = out[torch.from_numpy(rows).long().cuda()].cpu().numpy()
        got_l = lse[torch.from_numpy(rows).long().cuda()].cpu().numpy()
        assert np.abs(got_o - ro).max() <= gu.ATOL and np.abs(got_l - rlse).max() <= gu.ATOL
    # allocation-free entry: only out and out_lse are the caller's
    ob2, out2 = gu.guarded((T, H, D), torch.float32, G)
    lb2, lse2 = gu.guarded((T, H), torch.float32, G)
    pkv.paged_attention_varlen_noalloc(q, pool, table, cu, lens, w.max_query_len, w.max_seq_len,
                                       out=out2, out_lse=lse2, scale=w.scale, partition_size=256,
                                       dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert gu.guards_intact(ob2, out2.numel(), G) and gu.guards_intact(lb2, lse2.numel(), G)
