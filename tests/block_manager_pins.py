"""Pins of the reference block manager (``oracle/block_manager.py``).

Each pin is a plain function taking the module under test, so that the
mutation test can run the same battery against planted mistakes. They check
the oracle against things other than itself: the page's worked examples
(``tests/golden/block_tables.json``), counts that follow from the definitions
(references, free blocks, table lengths) and brute-force re-derivations of
slots from the tables.
"""
import json
import os
import random

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "block_tables.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def pin_page_logical_to_physical(bm):
    """Page 2's table example: logical blocks 1, 2, 3 live in physical blocks
    57, 1024, 233; a token's slot follows from that table."""
    g = _golden()["logical_to_physical_example"]
    nb = max(g) + 1
    order = g + [b for b in range(nb) if b not in g]
    m = bm.BlockManagerOracle(nb, 16, order)
    m.add_seq(0)
    slots, copies = m.append(0, 40)
    assert m.block_table(0) == g and copies == []
    assert slots[20] == 1024 * 16 + 4 and slots[39] == 233 * 16 + 7
    assert slots == [g[p // 16] * 16 + p % 16 for p in range(40)]


def pin_page_copy_on_write_tables(bm):
    """Page 2's copy-on-write diagram: after a fork, A = [7, 2] and
    B = [7, 6, 4] share physical block 7 (the prompt's block)."""
    g = _golden()
    order = [7, 2, 6, 4] + [b for b in range(8) if b not in (7, 2, 6, 4)]
    m = bm.BlockManagerOracle(8, 4, order)
    m.add_seq(0)
    m.append(0, 4)          # the prompt fills block 7
    m.fork(0, 1)            # B copies A's table only
    assert m.block_table(1) == [7] and m.num_free() == 7
    _, ca = m.append(0, 1)  # A diverges into a fresh block
    _, cb = m.append(1, 5)  # B diverges into two fresh blocks
    assert m.block_table(0) == g["cow_request_a"]
    assert m.block_table(1) == g["cow_request_b"]
    assert ca == [] and cb == []  # a full shared block is never written again
    assert m.ref[g["shared_physical_block"]] == 2


def pin_partial_shared_block_is_copied_once(bm):
    """Fork while the last block is half full: the first writer copies it,
    the other then owns the original alone and writes in place."""
    m = bm.BlockManagerOracle(6, 4)
    m.add_seq(0)
    m.append(0, 6)                      # blocks 0 (full), 1 (2 of 4)
    m.fork(0, 1)
    slots_a, copies_a = m.append(0, 1)
    assert copies_a == [(1, 2)] and slots_a == [2 * 4 + 2]
    assert m.block_table(0) == [0, 2] and m.block_table(1) == [0, 1]
    slots_b, copies_b = m.append(1, 1)
    assert copies_b == [] and slots_b == [1 * 4 + 2]
    assert m.ref == [2, 1, 1, 0, 0, 0]


def pin_free_returns_blocks_in_order(bm):
    m = bm.BlockManagerOracle(4, 2)
    m.add_seq(0)
    m.append(0, 3)          # blocks 0, 1
    m.add_seq(1)
    m.append(1, 1)          # block 2
    m.free_seq(0)           # 0 and 1 join the back of the queue
    assert list(m.free) == [3, 0, 1]
    m.add_seq(2)
    s, _ = m.append(2, 3)
    assert m.block_table(2) == [3, 0] and s == [6, 7, 0]


def pin_exhaustion_changes_nothing(bm):
    m = bm.BlockManagerOracle(3, 4)
    m.add_seq(0)
    m.append(0, 6)
    m.fork(0, 1)
    before = (m.block_table(0), m.block_table(1), list(m.free), list(m.ref))
    try:
        m.append(1, 7)      # needs a copy of block 1 plus one more block: 2 > 1 free
    except bm.OutOfBlocks:
        pass
    else:
        raise AssertionError("expected OutOfBlocks")
    assert (m.block_table(0), m.block_table(1), list(m.free), list(m.ref)) == before
    assert m.blocks_needed(1, 2) == 1 and m.blocks_needed(1, 3) == 2


def _check_invariants(m, store, hist):
    nb, bs = m.num_blocks, m.block_size
    refs = [0] * nb
    for sid, table in m.tables.items():
        assert len(table) == -(-m.lens[sid] // bs), "table length"
        for b in table:
            refs[b] += 1
    assert refs == m.ref, "reference counts"
    used = {b for t in m.tables.values() for b in t}
    assert set(m.free).isdisjoint(used) and len(set(m.free)) == len(m.free)
    assert len(m.free) + len(used) == nb, "every block is free or in use"
    # brute force: every live sequence reads back each of its tokens -- its
    # own, or the ones inherited from the sequence it was forked from
    for sid, length in m.lens.items():
        for pos in range(length):
            assert store.get(m.slot_of(sid, pos)) == (hist[sid][pos], pos), "token lost"


def pin_random_operations_keep_the_invariants(bm):
    """Random add / fork / append / free sequences: references equal the
    number of tables naming a block, every block is either free or used, and
    every token stays readable at the slot its table gives (copies carry
    shared tokens; a sequence never writes over another's token)."""
    rnd = random.Random(5)
    for trial in range(20):
        nb, bs = rnd.choice([(16, 2), (32, 4), (24, 16)])
        order = list(range(nb))
        rnd.shuffle(order)
        m = bm.BlockManagerOracle(nb, bs, order)
        store = {}   # slot -> (writer, position) of the token in it
        hist = {}    # sid -> writer of each of its positions
        next_id = 0
        for step in range(60):
            op = rnd.random()
            live = list(m.tables)
            if op < 0.2 or not live:
                m.add_seq(next_id)
                hist[next_id] = []
                next_id += 1
            elif op < 0.35:
                parent = rnd.choice(live)
                m.fork(parent, next_id)
                hist[next_id] = list(hist[parent])
                next_id += 1
            elif op < 0.85:
                sid = rnd.choice(live)
                n = rnd.randint(0, 2 * bs)
                try:
                    slots, copies = m.append(sid, n)
                except bm.OutOfBlocks:
                    continue
                for src, dst in copies:
                    for o in range(bs):
                        if src * bs + o in store:
                            store[dst * bs + o] = store[src * bs + o]
                base = len(hist[sid])
                for k, s in enumerate(slots):
                    store[s] = (sid, base + k)
                    hist[sid].append(sid)
            else:
                sid = rnd.choice(live)
                m.free_seq(sid)
                del hist[sid]
            _check_invariants(m, store, hist)


ALL_PINS = [
    pin_page_logical_to_physical,
    pin_page_copy_on_write_tables,
    pin_partial_shared_block_is_copied_once,
    pin_free_returns_blocks_in_order,
    pin_exhaustion_changes_nothing,
    pin_random_operations_keep_the_invariants,
]
