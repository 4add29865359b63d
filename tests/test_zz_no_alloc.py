"""The allocation-free attention entry point (needs a GB300).

pkv_paged_attention_varlen_noalloc is for callers that may not allocate
device memory -- an engine whose memory manager owns the whole GPU, a server
that must not call cudaMalloc while serving, a plugin handed only its inputs
and outputs. It takes its split-KV scratch from a fixed array inside the
library instead of a caller workspace. Its results must match the ordinary
entry point's, also on a second call in a row (the shared array keeps the
previous call's contents): both run the same kernels over the same
partitions, so they agree bit for bit. The file is named so that it runs last in a full
pass; it also passes on its own in a fresh process.
"""
import pytest
import torch

from paged_kv_cache_varlen_gb300 import binding as pkv
from paged_kv_cache_varlen_gb300 import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("partition_size", [-1, 256])
def test_noalloc_matches_workspace_entry_point_twice(partition_size):
    # decodes long enough to be split into several partitions, plus a prefill chunk
    w = wl.build("noalloc", [3000, 1500, 40, 2100, 600], [1, 1, 1, 1, 200], 32, 8, 128,
                 seed=301)
    dev = gu.DeviceStep(w)
    dev.write()
    assert dev.dev_status() == 0
    ref, ref_lse = dev.attend(partition_size=partition_size)
    assert dev.dev_status() == 0
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        pkv.paged_attention_varlen_noalloc(
            dev.q, dev.pool, dev.table, dev.cu, dev.lens, w.max_query_len, w.max_seq_len,
            out=out, out_lse=lse, scale=w.scale, partition_size=partition_size,
            dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.isfinite(out).all() and torch.isfinite(lse).all()
        # the same kernels over the same partitions: bit for bit the same
        assert torch.equal(out, ref) and torch.equal(lse, ref_lse)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # 512 requests x 32 heads x 32 partitions of partials need far more than 16 MiB
    B, H, D = 512, 32, 128
    need = pkv.attention_workspace_size(B, B, H, 8, D, 32 * 1024, 1024)
    assert need > 16 * 1024 * 1024
    q = torch.zeros((B, H, D), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((B, H, D), dtype=torch.float32, device="cuda")
    pool = torch.zeros((2, 8, 16, 8, D), dtype=torch.bfloat16, device="cuda")
    table = torch.zeros((B, 1), dtype=torch.int32, device="cuda")
    cu = torch.arange(B + 1, dtype=torch.int32, device="cuda")
    lens = torch.ones(B, dtype=torch.int32, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_attention_varlen_noalloc(q, pool, table, cu, lens, 1, 32 * 1024, out=out,
                                           partition_size=1024)
    assert e.value.status == 4
