"""The C ABI library: it loads, exports every symbol ``include/pkv.h``
declares, and its host-side checks reject bad arguments before touching the
GPU (CPU only: no kernel runs here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_varlen_gb300 import binding, build

    build.build()
    return binding.load_library()


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("pkv_kv_cache_write", "pkv_paged_attention_varlen", "pkv_lse_merge",
              "pkv_attention_workspace_size", "pkv_status_string", "pkv_abi_version"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version(lib):
    assert lib.pkv_abi_version() == 1
    assert lib.pkv_status_string(0) == b"ok"
    assert lib.pkv_status_string(4).startswith(b"workspace")


def test_workspace_size_arithmetic(lib):
    up = lambda x: -(-x // 256) * 256
    sched = 256  # prefill work tickets, always present
    # one partition: nothing to merge; only the tickets
    assert lib.pkv_attention_workspace_size(64, 64, 32, 8, 128, 512, -1) == sched
    assert lib.pkv_attention_workspace_size(64, 64, 32, 8, 128, 4096, 0) == sched
    # 4096 / 1024 = 4 partitions: [B][4][H][D] fp32 partials + [B][4][H] fp32 lse
    # + tickets, each piece 256-byte aligned
    rows = 64 * 4 * 32
    expect = up(rows * 128 * 4) + up(rows * 4) + sched
    assert lib.pkv_attention_workspace_size(64, 64, 32, 8, 128, 4096, -1) == expect
    assert lib.pkv_attention_workspace_size(64, 64, 32, 8, 128, 4096, 1024) == expect
    # explicit partition must be a multiple of 16
    assert lib.pkv_attention_workspace_size(64, 64, 32, 8, 128, 4096, 100) == 0
    # automatic partitions double until a request has at most 32 of them
    rows = 8 * 32 * 32            # 131072 tokens -> 4096-token partitions -> 32 parts
    assert lib.pkv_attention_workspace_size(8, 8, 32, 8, 128, 131072, -1) == \
        up(rows * 128 * 4) + up(rows * 4) + sched


def _attn(lib, **over):
    args = dict(out=16, out_lse=None, q=16, kv_pool=16, block_table=16, max_blocks=4, cu=16,
                seq_lens=16, num_seqs=1, num_tokens=1, max_query_len=1, max_seq_len=16,
                num_heads=4, num_kv_heads=2, head_dim=128, block_size=16, num_blocks=4,
                scale=0.125, partition_size=-1, workspace=None, workspace_bytes=0,
                dev_status=None, stream=None)
    args.update(over)
    return lib.pkv_paged_attention_varlen(*args.values())


@pytest.mark.parametrize("over,status", [
    ({"num_tokens": -1}, 1),
    ({"num_seqs": 0}, 1),
    ({"out": None}, 1),
    ({"q": None}, 1),
    ({"num_heads": 6, "num_kv_heads": 4}, 1),
    ({"max_query_len": 0}, 1),
    ({"max_seq_len": 0}, 1),
    ({"scale": 0.0}, 1),
    ({"scale": float("nan")}, 1),
    ({"q": 24}, 1),                      # not 16-byte aligned
    ({"head_dim": 96}, 2),
    ({"block_size": 8}, 2),
    ({"block_size": 512}, 2),
    ({"max_query_len": 2, "num_heads": 6, "num_kv_heads": 2}, 2),   # group 3 on the MMA path
    ({"partition_size": 100}, 1),
    ({"partition_size": -2}, 1),
    ({"max_seq_len": 4096, "partition_size": 512}, 4),             # needs workspace
])
def test_attention_rejects_before_launch(lib, over, status):
    assert _attn(lib, **over) == status


def test_empty_batch_is_a_no_op(lib):
    assert _attn(lib, num_tokens=0, out=None, q=None) == 0


@pytest.mark.parametrize("args,status", [
    ((16, 16, 16, 16, -1, 4, 16, 2, 128, None, None), 1),
    ((None, 16, 16, 16, 3, 4, 16, 2, 128, None, None), 1),
    ((16, 16, 16, 16, 3, 0, 16, 2, 128, None, None), 1),
    ((16, 16, 24, 16, 3, 4, 16, 2, 128, None, None), 1),
    ((16, 16, 16, 16, 3, 4, 16, 1, 4, None, None), 2),
    ((16, 16, 16, 16, 0, 4, 16, 2, 128, None, None), 0),
])
def test_kv_write_rejects_before_launch(lib, args, status):
    assert lib.pkv_kv_cache_write(*args) == status


@pytest.mark.parametrize("args,status", [
    ((16, None, 16, 16, 0, 4, 2, 128, None), 1),
    ((16, None, 16, 16, 2, 4, 2, 130, None), 2),
    ((16, None, 16, 16, 2, 4, 2, 1024, None), 2),
    ((None, None, 16, 16, 2, 4, 2, 128, None), 1),
    ((16, None, 16, 16, 2, 0, 2, 128, None), 0),
])
def test_lse_merge_rejects_before_launch(lib, args, status):
    assert lib.pkv_lse_merge(*args) == status


def test_binding_fails_loudly_without_library(tmp_path):
    from paged_kv_cache_varlen_gb300 import binding

    with pytest.raises(binding.PkvError):
        binding.load_library(str(tmp_path / "missing.so"))


def test_cascade_workspace_size_arithmetic(lib):
    up = lambda x: -(-x // 256) * 256
    B, H, Hkv, D = 256, 32, 8, 128

    def expect(splits, tail_parts):
        rows = (splits + 1) * B * H          # S prefix segments, then the tail
        size = up(rows * D * 4) + up(rows * 4) + up((B + 1) * 4)
        if tail_parts > 1:                   # the tail pass's own split-KV partials
            trows = B * tail_parts * H
            size += up(trows * D * 4) + up(trows * 4)
        return size + 256                    # prefill work tickets
    # 4 groups of 64 members, 2048-token prefixes: 64 queries per work item at
    # G = 4, so 4 x 1 x 8 = 32 items; ceil(148 / 32) = 5 key segments
    assert lib.pkv_cascade_workspace_size(B, 4, 64, 2048, 1024, H, Hkv, D) == expect(5, 1)
    # tails up to 3000 tokens split into 3 partitions of 1024
    assert lib.pkv_cascade_workspace_size(B, 4, 64, 2048, 3000, H, Hkv, D) == expect(5, 3)
    # no groups: one (empty) prefix slot and the tail
    assert lib.pkv_cascade_workspace_size(B, 0, 1, 0, 1024, H, Hkv, D) == expect(1, 1)
    # segments never outnumber the prefix's 128-key tiles (256 tokens: 2 tiles)
    assert lib.pkv_cascade_workspace_size(B, 1, 4, 256, 1024, H, Hkv, D) == expect(2, 1)
    # invalid sizes
    assert lib.pkv_cascade_workspace_size(0, 4, 64, 2048, 1024, H, Hkv, D) == 0
    assert lib.pkv_cascade_workspace_size(B, 4, 64, 2048, 1024, 30, Hkv, D) == 0


@pytest.mark.parametrize("args,status", [
    ((16, 16, 16, -1, 8, 16, 2, 128, None, None), 1),     # negative count
    ((16, 16, 16, 0, 8, 16, 2, 128, None, None), 0),      # nothing to copy
    ((None, 16, 16, 2, 8, 16, 2, 128, None, None), 1),    # no pool
    ((24, 16, 16, 2, 8, 16, 2, 128, None, None), 1),      # pool not 16-byte aligned
    ((16, None, 16, 2, 8, 16, 2, 128, None, None), 1),    # no source list
    ((16, 16, 16, 2, 0, 16, 2, 128, None, None), 1),      # empty pool
])
def test_copy_blocks_rejects_before_launch(lib, args, status):
    assert lib.pkv_copy_blocks(*args) == status
