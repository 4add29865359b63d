"""Shared-prefix (cascade) decode against the oracle (needs a GB300).

The cascade call must return what plain attention over each request's whole
context returns: prefix read once per group on the tensor cores, tails on
the decode kernel, partials merged by log-sum-exp. Cases: the 4 x 64
copy-on-write workload, plus groups of 1 and of more members than one tile
pair holds, a group with an empty prefix, requests in no group, different
prefix lengths, and an 8-way GQA shape.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_varlen_gb300 import binding as pkv
from paged_kv_cache_varlen_gb300 import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def run_cascade(w, dev, ci):
    out = torch.full((w.num_seqs, w.num_heads, w.head_dim), float("nan"), dtype=torch.float32,
                     device="cuda")
    lse = torch.full((w.num_seqs, w.num_heads), float("nan"), dtype=torch.float32, device="cuda")
    pkv.cascade_decode(dev.q, dev.pool, gu.i32_tensor(ci["group_starts"]),
                       gu.i32_tensor(ci["prefix_lens"]), gu.i32_tensor(ci["prefix_tables"]),
                       ci["max_group_size"], ci["max_prefix_len"], gu.i32_tensor(ci["tail_tables"]),
                       gu.i32_tensor(ci["tail_lens"]), ci["max_tail_len"], out=out, out_lse=lse,
                       scale=w.scale, dev_status=dev.status)
    return out, lse


def check(oracle, w, groups):
    ref_pool = oracle.kv_cache_write(w.pool, w.k_new, w.v_new, w.slot_mapping)
    dev = gu.DeviceStep(w)
    dev.write()
    ci = wl.cascade_inputs(w, groups)
    out, lse = run_cascade(w, dev, ci)
    assert dev.dev_status() == 0
    ref_o, ref_l = oracle.paged_attention(w.q, ref_pool, w.block_table, w.cu_seqlens, w.seq_lens,
                                          w.scale)
    gu.compare(out, lse, ref_o, ref_l)
    # and it agrees with the ordinary decode path
    out2, lse2 = dev.attend()
    assert dev.dev_status() == 0
    assert float((out - out2).abs().max()) <= gu.ATOL and float((lse - lse2).abs().max()) <= gu.ATOL


def test_prefix_cow_workload(oracle):
    w = wl.prefix_shared()
    check(oracle, w, wl.prefix_groups(w))


def test_mixed_groups(oracle):
    # groups of 1, 3 and 70 members (two work units), prefixes 16, 48 and 512
    # tokens, a group with an empty prefix, and 5 requests in no group
    sizes = [1, 3, 70, 4]
    prefixes = [16, 48, 512, 0]
    rng = np.random.default_rng(71)
    lens, sp, groups, first = [], [], [], 0
    for n, p in zip(sizes, prefixes):
        lens += list(p + rng.integers(1, 300, size=n, endpoint=True))
        if p:
            sp.append((list(range(first, first + n)), p))
        groups.append((first, n, p))
        first += n
    lens += list(rng.integers(1, 900, size=5, endpoint=True))
    b = len(lens)
    w = wl.build("cascade_mixed", lens, [1] * b, 32, 8, 128, 16, seed=72, shared_prefix=sp)
    check(oracle, w, groups)


def test_gqa8_head_dim_64(oracle):
    rng = np.random.default_rng(81)
    n, p = 40, 256
    lens = list(p + rng.integers(1, 200, size=n, endpoint=True))
    w = wl.build("cascade_g8", lens, [1] * n, 32, 4, 64, 16, seed=82,
                 shared_prefix=[(list(range(n)), p)])
    check(oracle, w, [(0, n, p)])


def test_long_prefixes_and_split_tails(oracle):
    """Tails longer than one 1024-token partition: the tail pass splits them
    and merges the pieces in its own merge grid before the prefix segments
    and the tail are merged; prefixes of 4096 and 1024 tokens (more key
    segments), plus requests in no group with long contexts."""
    rng = np.random.default_rng(91)
    sizes, prefixes = [6, 2], [4096, 1024]
    lens, sp, groups, first = [], [], [], 0
    for n, p in zip(sizes, prefixes):
        lens += list(p + rng.integers(1100, 3000, size=n, endpoint=True))
        sp.append((list(range(first, first + n)), p))
        groups.append((first, n, p))
        first += n
    lens += list(rng.integers(2500, 5000, size=3, endpoint=True))
    w = wl.build("cascade_long", lens, [1] * len(lens), 32, 8, 128, 16, seed=92,
                 shared_prefix=sp)
    ci = wl.cascade_inputs(w, groups)
    assert ci["max_tail_len"] > 1024
    check(oracle, w, groups)
