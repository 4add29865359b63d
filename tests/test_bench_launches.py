"""bench.py's count of kernel launches per attention call, on CPU, against the
kernels the one-metric ncu launch lists of each workload show (the KV write
is counted separately, once per step)."""
import functools
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from paged_kv_cache_varlen_gb300 import workloads as wl  # noqa: E402


@functools.lru_cache(maxsize=None)
def _workload(name):
    if name == "long_split_kv":
        # one request of the long-context shape (the count depends on the
        # partitions, not on the batch; the full batch's pool takes ~30 s to build)
        return wl.long_decode(poison=False, batch=1)
    return wl.CONFIGS[name](poison=False)


@pytest.mark.parametrize("name, cascade, expected", [
    ("llama3_8b_decode", False, 2),  # decode grid + split-KV merge grid
    ("long_split_kv", False, 2),     # decode grid + merge grid (eight warps a row)
    ("spec_verify", False, 3),       # order kernel + decode grid + merge grid
    ("mixed_step", False, 3),        # prefill grid + decode grid + merge grid
    ("prefill_chunks", False, 1),    # prefill grid alone: no request is short
    ("prefix_cow", False, 2),        # decode grid + merge grid
    ("prefix_cow", True, 3),         # prefix pass + tail decode + cascade merge
])
def test_attention_launches_match_the_launch_lists(name, cascade, expected):
    w = _workload(name)
    ci = wl.cascade_inputs(w, wl.prefix_groups(w)) if cascade else None
    assert bench.attention_launches(w, -1, ci) == expected


def test_order_kernel_only_for_small_several_query_batches():
    # one query per request: no order kernel; several queries: one, up to 256 requests
    one = wl.build("one", [100] * 8, [1] * 8, 32, 8, 128, seed=5)
    several = wl.build("several", [100] * 8, [3] * 8, 32, 8, 128, seed=5)
    many = wl.build("many", [100] * 257, [2] * 257, 32, 8, 128, seed=5)
    assert bench.attention_launches(one, 0, None) == 1
    assert bench.attention_launches(several, 0, None) == 2
    assert bench.attention_launches(many, 0, None) == 1
