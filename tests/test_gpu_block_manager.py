"""Block copies on the GPU and whole steps driven by the native block manager
(needs a GB300).

copy_blocks must reproduce the reference copy bit for bit. The end-to-end
test plays a small beam-search-like schedule -- prompts, forks, divergent
continuations that force copy-on-write of half-filled shared blocks, freed
beams -- with the native manager building every step; the GPU runs
copy_blocks, the KV write and attention through the C ABI, the host runs the
same steps through the oracle, and the outputs agree within the attention
tolerance.
"""
import numpy as np
import pytest
import torch

from oracle import block_manager as bmo
from paged_kv_cache_varlen_gb300 import binding as pkv
from paged_kv_cache_varlen_gb300 import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _pool(rng, nb, bs, hkv, d):
    return wl.to_bf16_bits(rng.standard_normal((2, nb, bs, hkv, d), dtype=np.float32))


def test_copy_blocks_bit_exact():
    rng = np.random.default_rng(41)
    nb, bs, hkv, d = 96, 16, 8, 128
    pool = _pool(rng, nb, bs, hkv, d)
    ids = rng.permutation(nb)
    src, dst = ids[:20].astype(np.int32), ids[20:40].astype(np.int32)
    want = bmo.apply_copies(pool, list(zip(src.tolist(), dst.tolist())))
    dev = gu.bf16_tensor(pool)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.copy_blocks(dev, gu.i32_tensor(src), gu.i32_tensor(dst), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(gu.to_numpy_bits(dev).reshape(pool.shape), want)


def test_copy_blocks_flags_bad_ids_and_copies_the_rest():
    rng = np.random.default_rng(42)
    nb, bs, hkv, d = 8, 16, 2, 64
    pool = _pool(rng, nb, bs, hkv, d)
    src = np.array([0, 1, 9], dtype=np.int32)
    dst = np.array([4, 5, 6], dtype=np.int32)
    want = bmo.apply_copies(pool, [(0, 4), (1, 5)])
    dev = gu.bf16_tensor(pool)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.copy_blocks(dev, gu.i32_tensor(src), gu.i32_tensor(dst), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == pkv.DEV_BAD_BLOCK
    assert np.array_equal(gu.to_numpy_bits(dev).reshape(pool.shape), want)


def test_beam_schedule_end_to_end(oracle):
    rng = np.random.default_rng(43)
    nb, bs, h, hkv, d = 64, 16, 8, 2, 64
    scale = 1.0 / np.sqrt(d)
    order = rng.permutation(nb).astype(np.int32)
    native = pkv.BlockManager(nb, bs, order)
    ref = bmo.BlockManagerOracle(nb, bs, order)
    pool_host = np.zeros((2, nb, bs, hkv, d), dtype=np.uint16)
    pool_dev = gu.bf16_tensor(pool_host)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    max_blocks = 16

    def step(seq_ids, num_new):
        nonlocal pool_host
        trial_out = [ref.append(s, n) for s, n in zip(seq_ids, num_new)]
        table, lens, cu, slots, src, dst = native.build_step(seq_ids, num_new, max_blocks)
        assert slots.tolist() == [x for o in trial_out for x in o[0]]
        copies = [c for o in trial_out for c in o[1]]
        assert list(zip(src.tolist(), dst.tolist())) == copies
        t = int(cu[-1])
        q = wl.to_bf16_bits(rng.standard_normal((t, h, d), dtype=np.float32))
        kn = wl.to_bf16_bits(rng.standard_normal((t, hkv, d), dtype=np.float32))
        vn = wl.to_bf16_bits(rng.standard_normal((t, hkv, d), dtype=np.float32))
        # host: the oracle's copy, write and attention
        pool_host = bmo.apply_copies(pool_host, copies)
        pool_host = oracle.kv_cache_write(pool_host, kn, vn, slots)
        ref_o, ref_l = oracle.paged_attention(q, pool_host, table, cu, lens, scale)
        # device: the same step through the C ABI
        if copies:
            pkv.copy_blocks(pool_dev, gu.i32_tensor(src), gu.i32_tensor(dst), dev_status=status)
        pkv.kv_cache_write(pool_dev, gu.bf16_tensor(kn), gu.bf16_tensor(vn), gu.i32_tensor(slots),
                           dev_status=status)
        out = torch.full((t, h, d), float("nan"), dtype=torch.float32, device="cuda")
        lse = torch.full((t, h), float("nan"), dtype=torch.float32, device="cuda")
        pkv.paged_attention_varlen(gu.bf16_tensor(q), pool_dev, gu.i32_tensor(table),
                                   gu.i32_tensor(cu), gu.i32_tensor(lens),
                                   int(np.max(num_new)), int(lens.max()), out=out, out_lse=lse,
                                   scale=scale, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        gu.compare(out, lse, ref_o, ref_l)
        return len(copies)

    for sid in (0, 1):
        native.add_seq(sid)
        ref.add_seq(sid)
    step([0, 1], [37, 20])            # prompts: half-filled last blocks
    for child, parent in ((2, 0), (3, 0), (4, 1)):
        native.fork(parent, child)
        ref.fork(parent, child)
    n_copies = 0
    beams = [0, 1, 2, 3, 4]
    for it in range(12):
        n_copies += step(beams, [1] * len(beams))
        if it == 5:                   # prune a beam, fork another
            native.free_seq(3)
            ref.free_seq(3)
            native.fork(2, 5)
            ref.fork(2, 5)
            beams = [0, 1, 2, 4, 5]
    assert n_copies >= 4              # the shared half-filled blocks were copied
    assert native.num_free() == ref.num_free()
