"""Host-side index checks of the debug mode (PKV_DEBUG_CHECKS=1), on CPU:
valid tables of every workload shape pass; each kind of bad entry the kernels
would skip and flag raises, naming the entry."""
import numpy as np
import pytest

from paged_kv_cache_varlen_gb300 import debug_checks as dc
from paged_kv_cache_varlen_gb300 import workloads as wl


def _args(w, **over):
    a = dict(num_tokens=w.num_tokens, max_query_len=w.max_query_len, max_seq_len=w.max_seq_len,
             num_blocks=w.num_blocks, block_size=w.block_size)
    a.update(over)
    return a


@pytest.mark.parametrize("name", ["tiny", "llama3_8b_decode", "spec_verify", "mixed_step",
                                  "prefill_chunks"])
def test_valid_tables_pass(name):
    w = wl.CONFIGS[name](poison=False)
    dc.check_attention_tables(w.cu_seqlens, w.seq_lens, w.block_table, **_args(w))
    dc.check_slot_mapping(w.slot_mapping, num_blocks=w.num_blocks, block_size=w.block_size)


@pytest.fixture(scope="module")
def small():
    return wl.build("dbg", [40, 300, 50, 77], [1, 1, 20, 0], 32, 8, 128, seed=301)


def test_block_id_outside_the_pool(small):
    w = small
    t = w.block_table.copy()
    t[1, 5] = w.num_blocks + 3
    with pytest.raises(ValueError, match=r"block_table\[1\]\[5\]"):
        dc.check_attention_tables(w.cu_seqlens, w.seq_lens, t, **_args(w))
    t = w.block_table.copy()
    t[2, 0] = -1
    with pytest.raises(ValueError, match=r"block_table\[2\]\[0\]"):
        dc.check_attention_tables(w.cu_seqlens, w.seq_lens, t, **_args(w))


def test_entries_past_the_context_and_empty_requests_are_not_read(small):
    w = small
    t = w.block_table.copy()
    nblk = -(-w.seq_lens // w.block_size)
    t[0, nblk[0]:] = -7          # past request 0's context
    t[3, :] = -7                 # request 3 has no query
    dc.check_attention_tables(w.cu_seqlens, w.seq_lens, t, **_args(w))


def test_lengths(small):
    w = small
    lens = w.seq_lens.copy()
    lens[2] = 5                  # shorter than its 20 queries
    with pytest.raises(ValueError, match="request 2"):
        dc.check_attention_tables(w.cu_seqlens, lens, w.block_table, **_args(w))
    with pytest.raises(ValueError, match="max_seq_len"):
        dc.check_attention_tables(w.cu_seqlens, w.seq_lens, w.block_table,
                                  **_args(w, max_seq_len=100))
    with pytest.raises(ValueError, match="max_query_len"):
        dc.check_attention_tables(w.cu_seqlens, w.seq_lens, w.block_table,
                                  **_args(w, max_query_len=8))
    cu = w.cu_seqlens.copy()
    cu[2], cu[3] = cu[3], cu[2]
    with pytest.raises(ValueError, match="decreases"):
        dc.check_attention_tables(cu, w.seq_lens, w.block_table, **_args(w))
    with pytest.raises(ValueError, match="num_tokens"):
        dc.check_attention_tables(w.cu_seqlens, w.seq_lens, w.block_table,
                                  **_args(w, num_tokens=w.num_tokens + 1))
    short = w.block_table[:, :2]
    with pytest.raises(ValueError, match="table row"):
        dc.check_attention_tables(w.cu_seqlens, w.seq_lens, short, **_args(w))


def test_key_ranges(small):
    w = small
    ks = np.zeros(4, dtype=np.int32)
    qs = (w.seq_lens - np.diff(w.cu_seqlens)).astype(np.int32)
    dc.check_attention_tables(w.cu_seqlens, w.seq_lens, w.block_table, **_args(w),
                              key_start=ks, query_start=qs)
    qs[1] = -1
    with pytest.raises(ValueError, match="negative"):
        dc.check_attention_tables(w.cu_seqlens, w.seq_lens, w.block_table, **_args(w),
                                  key_start=ks, query_start=qs)


def test_slots(small):
    w = small
    s = w.slot_mapping.copy()
    s[0] = -1                    # padding: skipped
    dc.check_slot_mapping(s, num_blocks=w.num_blocks, block_size=w.block_size)
    s[3] = w.num_blocks * w.block_size
    with pytest.raises(ValueError, match=r"slot_mapping\[3\]"):
        dc.check_slot_mapping(s, num_blocks=w.num_blocks, block_size=w.block_size)


def test_switch(monkeypatch):
    monkeypatch.delenv("PKV_DEBUG_CHECKS", raising=False)
    assert not dc.enabled()
    monkeypatch.setenv("PKV_DEBUG_CHECKS", "1")
    assert dc.enabled()


@pytest.mark.parametrize("name", ["tiny", "spec_verify", "mixed_step"])
def test_append_slots_of_valid_steps_pass(name):
    w = wl.CONFIGS[name](poison=False)
    dc.check_append_slots(w.cu_seqlens, w.seq_lens, w.block_table, w.slot_mapping,
                          block_size=w.block_size)


def test_append_slot_elsewhere_in_the_pool(small):
    w = small
    s = w.slot_mapping.copy()
    s[1] = -1                    # a skipped token is allowed
    dc.check_append_slots(w.cu_seqlens, w.seq_lens, w.block_table, s, block_size=w.block_size)
    s[2] = (s[2] + w.block_size) % (w.num_blocks * w.block_size)   # another block's slot
    with pytest.raises(ValueError, match=r"slot_mapping\[2\]"):
        dc.check_append_slots(w.cu_seqlens, w.seq_lens, w.block_table, s,
                              block_size=w.block_size)
