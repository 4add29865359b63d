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


@pytest.mark.parametrize("head_dim, limit", [(128, 8575), (64, 33151)])
def test_prefill_request_limit(lib, head_dim, limit):
    # a call with prefill work (max_query_len above 32 / G) keeps the prefill
    # kernel's work list in shared memory: at the limit the call gets past
    # that check (and stops at the missing workspace), one request more is
    # unsupported; decode-only calls are not limited by it
    big = dict(max_query_len=64, max_seq_len=64, head_dim=head_dim)
    assert _attn(lib, num_seqs=limit, num_tokens=limit, **big) == 4
    assert _attn(lib, num_seqs=limit + 1, num_tokens=limit + 1, **big) == 2
    assert _attn(lib, num_seqs=limit + 1, num_tokens=limit + 1, head_dim=head_dim,
                 max_seq_len=4096, partition_size=0) == 4


def test_partition_count_limit(lib):
    # 16-token partitions: 65535 of them per request is the most the decode
    # grid takes (the call then stops at the missing workspace); one more is
    # unsupported, and the workspace query gives 0 for it
    at, over = 65535 * 16, 65535 * 16 + 1
    assert _attn(lib, max_seq_len=at, max_blocks=at // 16, partition_size=16) == 4
    assert _attn(lib, max_seq_len=over, max_blocks=at // 16 + 1, partition_size=16) == 2
    assert lib.pkv_attention_workspace_size(1, 1, 4, 2, 128, at, 16) > 0
    assert lib.pkv_attention_workspace_size(1, 1, 4, 2, 128, over, 16) == 0


def _append(lib, **over):
    args = dict(out=16, out_lse=None, q=16, kv_pool=16, k_new=16, v_new=16, slot_mapping=16,
                block_table=16, max_blocks=4, cu=16, seq_lens=16, num_seqs=1, num_tokens=1,
                max_query_len=1, max_seq_len=16, num_heads=4, num_kv_heads=2, head_dim=128,
                block_size=16, num_blocks=4, scale=0.125, partition_size=-1, workspace=None,
                workspace_bytes=0, dev_status=None, stream=None)
    args.update(over)
    return lib.pkv_paged_attention_varlen_append(*args.values())


@pytest.mark.parametrize("over,status", [
    ({"k_new": None}, 1),
    ({"slot_mapping": None}, 1),
    ({"v_new": 24}, 1),                  # not 16-byte aligned
    ({"q": None}, 1),                    # the attention's own checks, before the write
    ({"head_dim": 96}, 2),
    ({}, 4),                             # every argument valid: stops at the missing workspace
])
def test_append_rejects_before_launch(lib, over, status):
    assert _append(lib, **over) == status


def test_append_empty_batch_is_a_no_op(lib):
    assert _append(lib, num_tokens=0, out=None, q=None, k_new=None) == 0


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
        rows = (splits + 1) * B * H          # the tail, then S prefix segments
        size = up(rows * D * 4) + up(rows * 4)
        if tail_parts > 1:                   # the tail pass's own split-KV partials
            trows = B * tail_parts * H
            size += up(trows * D * 4) + up(trows * 4)
        return size + 256                    # prefill work tickets
    # 4 groups of 64 members, 2048-token prefixes: 64 queries per work item at
    # G = 4, so 4 x 1 x 8 = 32 items; ceil(30 / 32) = 1 key segment (the
    # prefix pass takes about a fifth of the SMs, beside the tails)
    assert lib.pkv_cascade_workspace_size(B, 4, 64, 2048, 1024, H, Hkv, D) == expect(1, 1)
    # tails up to 3000 tokens split into 3 partitions of 1024
    assert lib.pkv_cascade_workspace_size(B, 4, 64, 2048, 3000, H, Hkv, D) == expect(1, 3)
    # one small group: ceil(30 / 8) = 4 segments of the 16 tiles
    assert lib.pkv_cascade_workspace_size(B, 1, 64, 2048, 1024, H, Hkv, D) == expect(4, 1)
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


# On a host without a GPU, the first CUDA step of a call that passed every
# host-side check fails with PKV_ERR_CUDA (3). A rejection status other than 3
# therefore shows that the call stopped before touching CUDA, i.e. before it
# could enqueue anything.

def _cascade(lib, **over):
    args = dict(out=256, out_lse=None, q=256, kv_pool=256, num_prefix_groups=1,
                group_starts=256, prefix_lens=256, prefix_tables=256, max_prefix_blocks=4,
                max_group_size=8, max_prefix_len=64, tail_tables=256, max_tail_blocks=4,
                tail_lens=256, max_tail_len=64, num_seqs=8, num_heads=32, num_kv_heads=8,
                head_dim=128, block_size=16, num_blocks=64, scale=0.088, workspace=256,
                workspace_bytes=1 << 30, dev_status=None, stream=None)
    args.update(over)
    return lib.pkv_cascade_decode(*args.values())


@pytest.mark.parametrize("over,status", [
    ({"head_dim": 96}, 2),            # rejected before the first launch
    ({"block_size": 8}, 2),
    ({"out": None}, 1),
    ({"workspace_bytes": 1024}, 4),
    ({"num_prefix_groups": 8576, "num_seqs": 8576}, 2),   # prefix pass work list too large
    ({}, 3),                          # every check passes: the first CUDA step fails here
])
def test_cascade_rejects_before_any_launch(lib, over, status):
    assert _cascade(lib, **over) == status


def _noalloc(lib, **over):
    args = dict(out=256, out_lse=None, q=256, kv_pool=256, block_table=256, max_blocks=512,
                cu=256, seq_lens=256, num_seqs=1, num_tokens=1, max_query_len=1,
                max_seq_len=8192, num_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                num_blocks=1024, scale=0.088, partition_size=-1, dev_status=None, stream=None)
    args.update(over)
    return lib.pkv_paged_attention_varlen_noalloc(*args.values())


@pytest.mark.parametrize("over,status", [
    ({"out": None}, 1),
    ({"q": None}, 1),
    ({"head_dim": 96}, 2),
    ({"num_tokens": 0, "out": None}, 0),   # an empty batch touches nothing
    # bad arguments are reported as such even when the sizes are beyond the scratch
    ({"out": None, "num_seqs": 4096, "num_tokens": 4096}, 1),
])
def test_noalloc_checks_arguments_before_its_scratch(lib, over, status):
    assert _noalloc(lib, **over) == status


def test_noalloc_scratch_boundary(lib):
    """16 MiB of built-in scratch: at 32 heads, D = 128 and 8 automatic
    1024-token partitions a request needs 8 * 32 * (128 + 1) * 4 bytes of
    partials, so 127 requests fit and 128 do not."""
    per_req = 8 * 32 * 128 * 4 + 8 * 32 * 4
    assert lib.pkv_attention_workspace_size(127, 127, 32, 8, 128, 8192, -1) == \
        127 * per_req + 256 <= 16 << 20
    assert lib.pkv_attention_workspace_size(128, 128, 32, 8, 128, 8192, -1) > 16 << 20
    # 127 passes the size check (and then fails at the first CUDA step on a
    # host without a GPU); 128 is rejected by it
    assert _noalloc(lib, num_seqs=127, num_tokens=127) == 3
    assert _noalloc(lib, num_seqs=128, num_tokens=128) == 4


def _range(lib, **over):
    args = dict(out=256, out_lse=None, q=256, kv_pool=256, block_table=256, max_blocks=4,
                cu=256, seq_lens=256, key_start=256, query_start=256, num_seqs=1, num_tokens=4,
                max_query_len=4, max_seq_len=2, num_heads=32, num_kv_heads=8, head_dim=128,
                block_size=16, num_blocks=8, scale=0.088, partition_size=-1, workspace=256,
                workspace_bytes=1 << 20, dev_status=None, stream=None)
    args.update(over)
    return lib.pkv_paged_attention_varlen_range(*args.values())


@pytest.mark.parametrize("over,status", [
    ({"key_start": None}, 1),
    ({"query_start": None}, 1),
    ({"max_seq_len": 0}, 1),
    ({"head_dim": 96}, 2),
    ({"workspace": None}, 4),
    ({"num_tokens": 0, "key_start": None}, 0),
    ({}, 3),          # a range may hold fewer keys than queries: accepted
])
def test_range_rejects_before_launch(lib, over, status):
    assert _range(lib, **over) == status
