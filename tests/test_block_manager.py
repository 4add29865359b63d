"""The native block manager (C++ behind the C ABI) against the reference
block manager of ``oracle/`` (CPU only: no CUDA call is involved).

Random operation sequences (add, fork, append, free, whole-batch steps) run
on both; every slot, copy, table, length, reference count and free count
must be identical, including the all-or-nothing refusals when the pool runs
out.
"""
import copy
import random

import numpy as np
import pytest

from oracle import block_manager as bmo
from paged_kv_cache_varlen_gb300 import binding as pkv

NO_BLOCKS = 5


def _same_state(native, ref):
    assert native.num_free() == ref.num_free()
    for b in range(ref.num_blocks):
        assert native.refcount(b) == ref.ref[b]
    for sid in ref.tables:
        assert native.block_table(sid) == ref.block_table(sid)
        assert native.seq_len(sid) == ref.seq_len(sid)


def test_page_copy_on_write_example():
    order = [7, 2, 6, 4, 0, 1, 3, 5]
    m = pkv.BlockManager(8, 4, order)
    m.add_seq(0)
    m.append(0, 4)
    m.fork(0, 1)
    m.append(0, 1)
    m.append(1, 5)
    assert m.block_table(0) == [7, 2] and m.block_table(1) == [7, 6, 4]
    assert m.refcount(7) == 2 and m.num_free() == 4


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_match_the_reference(seed):
    rnd = random.Random(100 + seed)
    nb, bs = rnd.choice([(16, 2), (40, 4), (24, 16), (64, 8)])
    order = list(range(nb))
    rnd.shuffle(order)
    native = pkv.BlockManager(nb, bs, order)
    ref = bmo.BlockManagerOracle(nb, bs, order)
    next_id = 0
    for step in range(300):
        live = list(ref.tables)
        op = rnd.random()
        if op < 0.15 or not live:
            native.add_seq(next_id)
            ref.add_seq(next_id)
            next_id += 1
        elif op < 0.3:
            parent = rnd.choice(live)
            native.fork(parent, next_id)
            ref.fork(parent, next_id)
            next_id += 1
        elif op < 0.6:
            sid = rnd.choice(live)
            n = rnd.randint(0, 3 * bs)
            try:
                want = ref.append(sid, n)
            except bmo.OutOfBlocks:
                with pytest.raises(pkv.PkvError) as e:
                    native.append(sid, n)
                assert e.value.status == NO_BLOCKS
            else:
                assert native.append(sid, n) == want
        elif op < 0.9:
            batch = rnd.sample(live, rnd.randint(1, len(live)))
            new = [rnd.randint(0, 2 * bs) for _ in batch]
            trial = copy.deepcopy(ref)
            try:
                out = [trial.append(s, n) for s, n in zip(batch, new)]
            except bmo.OutOfBlocks:
                with pytest.raises(pkv.PkvError) as e:
                    native.build_step(batch, new, max_blocks=nb)
                assert e.value.status == NO_BLOCKS
            else:
                ref = trial
                table, lens, cu, slots, src, dst = native.build_step(batch, new, max_blocks=nb)
                assert slots.tolist() == [s for o in out for s in o[0]]
                assert list(zip(src.tolist(), dst.tolist())) == [c for o in out for c in o[1]]
                assert cu.tolist() == [0] + np.cumsum(new).tolist()
                for i, sid in enumerate(batch):
                    t = ref.block_table(sid)
                    assert table[i, :len(t)].tolist() == t and (table[i, len(t):] == -1).all()
                    assert lens[i] == ref.seq_len(sid)
        else:
            sid = rnd.choice(live)
            native.free_seq(sid)
            ref.free_seq(sid)
        _same_state(native, ref)


def test_rejections():
    m = pkv.BlockManager(4, 4)
    m.add_seq(1)
    for call in (lambda: m.add_seq(1), lambda: m.fork(9, 2), lambda: m.fork(1, 1),
                 lambda: m.free_seq(9), lambda: m.append(9, 1),
                 lambda: m.build_step([1, 1], [1, 1], 4), lambda: m.build_step([1], [17], 4)):
        with pytest.raises(pkv.PkvError) as e:
            call()
        assert e.value.status == 1
    with pytest.raises(pkv.PkvError):
        pkv.BlockManager(4, 4, free_order=[0, 1, 1, 2])
    with pytest.raises(pkv.PkvError) as e:
        m.append(1, 17)
    assert e.value.status == NO_BLOCKS and m.num_free() == 4 and m.seq_len(1) == 0
