"""The combined KV write and attention call (GPU): the same pool and the same
outputs, bit for bit, as the KV write followed by the attention call, for
batches whose decode grid starts early (one-query decodes, split and unsplit;
several-query requests beyond the longest-first limit) and for those that wait
as the separate calls do (a longest-first verification batch, a mixed step);
and the outputs match the oracle."""
import numpy as np
import pytest
import torch

from paged_kv_cache_varlen_gb300 import binding as pkv
from paged_kv_cache_varlen_gb300 import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _append(dev, partition_size=-1):
    w = dev.w
    out = torch.full(tuple(dev.q.shape), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full(tuple(dev.q.shape[:2]), float("nan"), dtype=torch.float32, device="cuda")
    pkv.paged_attention_varlen_append(
        dev.q, dev.pool, dev.k_new, dev.v_new, dev.slots, dev.table, dev.cu, dev.lens,
        w.max_query_len, w.max_seq_len, out=out, out_lse=lse, scale=w.scale,
        partition_size=partition_size, dev_status=dev.status)
    return out, lse


def _batches():
    rng = np.random.default_rng(250)
    dec = rng.integers(40, 4000, size=48)
    many = 300  # several-query requests beyond the longest-first limit: early, unordered
    q_many = rng.integers(1, 4, size=many, endpoint=True)
    return {
        "decode": wl.build("ap_decode", dec, [1] * 48, 32, 8, 128, seed=251),
        "decode_d64": wl.build("ap_d64", dec[:16], [1] * 16, 16, 4, 64, seed=252),
        "verify_many": wl.build("ap_many", q_many + rng.integers(0, 600, size=many), q_many,
                                32, 8, 128, seed=253),
        "verify_ordered": wl.build("ap_ord", [900, 40, 2500, 7, 1300], [3, 1, 8, 7, 2],
                                   32, 8, 128, seed=254),
        "mixed": wl.build("ap_mixed", [3000, 600, 1700, 300], [1, 200, 1, 300], 32, 8, 128,
                          seed=255),
    }


@pytest.fixture(scope="module")
def batches():
    return _batches()


@pytest.mark.parametrize("name", ["decode", "decode_d64", "verify_many", "verify_ordered",
                                  "mixed"])
@pytest.mark.parametrize("partition_size", [-1, 64])
def test_append_equals_write_then_attend(oracle, batches, name, partition_size):
    w = batches[name]
    sep = gu.DeviceStep(w)
    sep.write()
    ref_out, ref_lse = sep.attend(partition_size=partition_size)
    assert sep.dev_status() == 0
    one = gu.DeviceStep(w)
    out, lse = _append(one, partition_size=partition_size)
    assert one.dev_status() == 0
    assert torch.equal(one.pool.view(torch.int16), sep.pool.view(torch.int16))
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    if partition_size == -1:
        ref_pool = oracle.kv_cache_write(w.pool, w.k_new, w.v_new, w.slot_mapping)
        ro, rl = oracle.paged_attention(w.q, ref_pool, w.block_table, w.cu_seqlens, w.seq_lens,
                                        w.scale)
        gu.compare(out, lse, ro, rl)


def test_append_back_to_back_steps(batches):
    """Calls one after another on one stream (each step's decode grid starting
    during the next KV write's predecessor): the same as separate calls."""
    w = batches["decode"]
    sep, one = gu.DeviceStep(w), gu.DeviceStep(w)
    outs_sep, outs_one = [], []
    for _ in range(3):
        sep.write()
        outs_sep.append(sep.attend())
        outs_one.append(_append(one))
    assert sep.dev_status() == 0 and one.dev_status() == 0
    for (a, la), (b, lb) in zip(outs_sep, outs_one):
        assert torch.equal(a, b) and torch.equal(la, lb)
