"""GPU edge cases (needs a GB300): split-KV partition sizes, ragged tails,
GQA group sizes, head_dim 64, larger blocks, short query chunks, the
invariants the oracle is pinned to (block permutation, copy-on-write
aliasing, length-1 contexts), device-side error bits and the public
log-sum-exp merge."""
import json
import math
import os

import numpy as np
import pytest
import torch

from paged_kv_cache_varlen_gb300 import binding as pkv
from paged_kv_cache_varlen_gb300 import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _run_and_check(oracle, w, partition_size=-1, rows=None):
    ref_pool = oracle.kv_cache_write(w.pool, w.k_new, w.v_new, w.slot_mapping)
    dev = gu.DeviceStep(w)
    dev.write()
    out, lse = dev.attend(partition_size=partition_size)
    assert dev.dev_status() == 0
    ref_o, ref_l = oracle.paged_attention(w.q, ref_pool, w.block_table, w.cu_seqlens, w.seq_lens,
                                          w.scale, rows=rows)
    gu.compare(out, lse, ref_o, ref_l, rows=rows)
    return dev, out, lse


@pytest.mark.parametrize("partition_size", [0, 16, 48, 128, 512, 2048, -1])
def test_decode_partition_sizes(oracle, partition_size):
    w = wl.build("parts", [1, 15, 16, 17, 511, 512, 513, 1500, 3001], [1] * 9, 32, 8, 128,
                 seed=201)
    _run_and_check(oracle, w, partition_size)


def test_one_partition_equals_no_split_bitwise():
    w = wl.build("onepart", [100, 700, 1023], [1, 1, 1], 32, 8, 128, seed=202)
    dev = gu.DeviceStep(w)
    dev.write()
    a = dev.attend(partition_size=0)
    b = dev.attend(partition_size=1024)   # every context fits one partition
    assert dev.dev_status() == 0
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("H,Hkv", [(32, 8), (8, 8), (32, 32), (32, 1), (16, 8), (64, 8), (4, 2)])
@pytest.mark.parametrize("D", [64, 128])
def test_group_sizes_and_head_dims_decode(oracle, H, Hkv, D):
    w = wl.build("gqa", [1, 33, 300, 1111], [1, 1, 1, 1], H, Hkv, D, seed=203 + H + Hkv + D)
    _run_and_check(oracle, w, 256)


@pytest.mark.parametrize("H,Hkv", [(32, 8), (8, 8), (32, 1), (16, 8), (8, 2)])
@pytest.mark.parametrize("D", [64, 128])
def test_group_sizes_and_head_dims_prefill(oracle, H, Hkv, D):
    w = wl.build("gqa_pre", [300, 40, 1, 257], [200, 40, 1, 17], H, Hkv, D, seed=204 + H + D)
    _run_and_check(oracle, w)


@pytest.mark.parametrize("BS", [16, 32, 64, 256])
def test_block_sizes(oracle, BS):
    w = wl.build("bs", [5, 77, 400, 1030], [1, 1, 70, 3], 32, 8, 128, block_size=BS, seed=205 + BS)
    _run_and_check(oracle, w, 128)


@pytest.mark.parametrize("qlens", [[2, 3, 4, 5, 6, 7, 8, 2], [33, 31, 1, 64, 65, 127, 129, 2]])
def test_short_query_chunks(oracle, qlens):
    """Speculative-verify sized chunks and chunk lengths around the 32-query
    tile, each over a cached prior context, mixed with decodes."""
    prior = [0, 5, 16, 100, 1000, 17, 4095, 64]
    L = [p + q for p, q in zip(prior, qlens)]
    w = wl.build("short", L, qlens, 32, 8, 128, seed=206 + sum(qlens))
    _run_and_check(oracle, w)


@pytest.mark.parametrize("H,Hkv,D", [(32, 8, 128), (32, 4, 128), (8, 8, 64), (32, 2, 128),
                                     (32, 1, 64)])
def test_verification_steps_around_the_decode_cutoff(oracle, H, Hkv, D):
    """Requests of a few queries run on the decode kernel while their
    (query, head) rows fit two 16-row MMA subgroups (q <= 32 / G), and on
    the prefill kernel beyond: every q from 1 to one past the cutoff, over
    prior contexts from empty to several blocks."""
    G = H // Hkv
    cut = max(1, 32 // G)
    qlens = list(range(1, cut + 2))
    prior = [(37 * k) % 300 for k in range(len(qlens))]
    L = [p + q for p, q in zip(prior, qlens)]
    w = wl.build("verify", L, qlens, H, Hkv, D, seed=260 + G + D)
    _run_and_check(oracle, w)


@pytest.mark.parametrize("case", ["decode_heavy", "prefill_heavy", "empty_requests"])
def test_mixed_batches_at_the_ends_of_the_sm_split(oracle, case):
    """With decodes in the call the prefill grid keeps about its share of the
    SMs and its other CTAs leave at once: long decodes beside one small chunk
    (the share clamps to a single prefill CTA), one long chunk beside a single
    short decode, and requests of no query beside both kinds. The results do
    not depend on the split."""
    if case == "decode_heavy":
        L, q = [8000, 7000, 6000, 5000, 4000, 3000, 2000, 1000] * 4 + [200], [1] * 32 + [40]
    elif case == "prefill_heavy":
        L, q = [2500, 300], [1000, 1]
    else:
        L, q = [300, 50, 1000, 700, 64], [0, 40, 1, 0, 3]
    w = wl.build("split_" + case, L, q, 32, 8, 128, seed=219 + len(L))
    _run_and_check(oracle, w)


@pytest.mark.parametrize("n", [64, 256, 300])
def test_verification_batches_in_and_out_of_longest_first_order(oracle, n):
    """Decode-only batches with several-query requests run longest context
    first when they have at most 256 requests (and in request order beyond):
    lengths with ties, both sides of the limit."""
    rng = np.random.default_rng(230 + n)
    q = rng.integers(1, 8, size=n, endpoint=True)
    L = q + rng.choice([0, 17, 300, 300, 1024, 2000], size=n)
    w = wl.build("order", L, q, 32, 8, 128, seed=231 + n)
    _run_and_check(oracle, w)


@pytest.mark.parametrize("H,Hkv", [(32, 8), (8, 8)])
def test_verification_batches_head_dim_64(oracle, H, Hkv):
    """The longest-first decode grid at head_dim 64: G = 4 (up to 8 queries,
    32 rows a request) and G = 1 (up to 32 queries, two 16-row subgroups),
    with one-query requests long enough to be split among them."""
    G = H // Hkv
    dmq = max(1, 32 // G)
    rng = np.random.default_rng(240 + G)
    n = 48
    q = rng.integers(1, dmq, size=n, endpoint=True)
    L = q + rng.choice([0, 5, 200, 700, 1500, 3000], size=n)
    w = wl.build("verify64", L, q, H, Hkv, 64, seed=241 + G)
    _run_and_check(oracle, w)


def test_full_prefill_without_prior_context(oracle):
    w = wl.build("fresh", [1, 2, 127, 128, 129, 600], [1, 2, 127, 128, 129, 600], 32, 8, 128,
                 seed=207)
    _run_and_check(oracle, w)


def test_length_one_context_returns_v_exactly():
    w = wl.build("l1", [1, 1, 1], [1, 1, 1], 32, 8, 128, seed=208)
    dev = gu.DeviceStep(w)
    dev.write()
    out, _ = dev.attend()
    assert dev.dev_status() == 0
    G = 4
    v = wl.bf16_bits_to_f32(w.v_new)
    ref = np.repeat(v, G, axis=1)          # head h reads kv head h // G
    assert np.array_equal(out.cpu().numpy(), ref)


@pytest.mark.parametrize("qlen", [1, 300])
def test_block_permutation_is_bitwise_invisible(qlen):
    w = wl.build("perm", [1400, 333], [1, qlen], 32, 8, 128, seed=209, pool_factor=1.5)
    dev = gu.DeviceStep(w)
    dev.write()
    out, lse = dev.attend()
    perm = np.random.default_rng(210).permutation(w.num_blocks)
    perm_t = torch.from_numpy(perm).cuda()
    pool2 = torch.empty_like(dev.pool)
    pool2[:, perm_t] = dev.pool
    bt2 = np.where(w.block_table >= 0, perm[np.maximum(w.block_table, 0)], -1)
    out2, lse2 = dev.attend(pool=pool2, table=gu.i32_tensor(bt2))
    assert dev.dev_status() == 0
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_copy_on_write_aliasing_is_bitwise_invisible():
    """The page's copy-on-write example: requests A = [7, 2] and B = [7, 6, 4]
    share physical block 7; a private copy of it for B changes nothing."""
    with open(os.path.join(GOLDEN, "block_tables.json")) as f:
        g = json.load(f)
    a_tab, b_tab = g["cow_request_a"], g["cow_request_b"]
    BS, H, Hkv, D, NB = 16, 32, 8, 128, 12
    rng = np.random.default_rng(211)
    pool = wl.to_bf16_bits(rng.standard_normal((2, NB, BS, Hkv, D), dtype=np.float32))
    q = wl.to_bf16_bits(rng.standard_normal((2, H, D), dtype=np.float32))
    lens = np.array([2 * BS, 3 * BS - 5], np.int32)
    cu = np.array([0, 1, 2], np.int32)

    def run(pool_np, table):
        out = torch.empty((2, H, D), dtype=torch.float32, device="cuda")
        lse = torch.empty((2, H), dtype=torch.float32, device="cuda")
        pkv.paged_attention_varlen(gu.bf16_tensor(q), gu.bf16_tensor(pool_np),
                                   gu.i32_tensor(np.array(table, np.int32)), gu.i32_tensor(cu),
                                   gu.i32_tensor(lens), 1, int(lens.max()), out=out, out_lse=lse)
        return out, lse

    o1, l1 = run(pool, [a_tab + [-1], b_tab])
    pool2 = pool.copy()
    pool2[:, 9] = pool[:, g["shared_physical_block"]]
    o2, l2 = run(pool2, [a_tab + [-1], [9] + b_tab[1:]])
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_nan_poisoned_free_slots_never_leak(oracle):
    """Unwritten slots of every partial last block hold bf16 NaN (the
    workload generator poisons them); outputs must stay finite and exact."""
    w = wl.build("nan", [17, 31, 130, 260], [1, 20, 130, 3], 32, 8, 128, seed=212)
    assert np.any(w.pool == wl.BF16_NAN)
    _run_and_check(oracle, w)


def test_empty_batch_is_a_no_op():
    out = torch.full((0, 32, 128), 1.0, device="cuda")
    q = torch.zeros((0, 32, 128), dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros((2, 4, 16, 8, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    cu = torch.zeros(2, dtype=torch.int32, device="cuda")
    lens = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.paged_attention_varlen(q, pool, bt, cu, lens, 1, 1, out=out)
    slots = torch.zeros(0, dtype=torch.int32, device="cuda")
    kn = torch.zeros((0, 8, 128), dtype=torch.bfloat16, device="cuda")
    pkv.kv_cache_write(pool, kn, kn, slots)
    torch.cuda.synchronize()


def test_device_errors_set_status_bits_and_spare_other_requests(oracle):
    w = wl.build("bad", [40, 300, 50], [1, 1, 20], 32, 8, 128, seed=213)
    ref_pool = oracle.kv_cache_write(w.pool, w.k_new, w.v_new, w.slot_mapping)
    ref_o, _ = oracle.paged_attention(w.q, ref_pool, w.block_table, w.cu_seqlens, w.seq_lens,
                                      w.scale)
    dev = gu.DeviceStep(w)
    dev.write()
    assert dev.dev_status() == 0
    # a block id outside the pool in request 1 (decode) and request 2 (prefill)
    bad = w.block_table.copy()
    bad[1, 3] = w.num_blocks + 5
    bad[2, 1] = -7
    out, _ = dev.attend(table=gu.i32_tensor(bad))
    assert dev.dev_status() & gu.pkv.DEV_BAD_BLOCK
    got = out.cpu().numpy()
    assert np.max(np.abs(got[0] - ref_o[0])) <= gu.ATOL   # request 0 untouched
    # a context shorter than its query chunk
    dev.status.zero_()
    lens = w.seq_lens.copy()
    lens[2] = 5
    dev.attend(lens=gu.i32_tensor(lens))
    assert dev.dev_status() & gu.pkv.DEV_BAD_LENGTHS
    # a verification request longer than the max_query_len the call was given
    wv = wl.build("badq", [40, 300], [1, 3], 32, 8, 128, seed=215)
    ref_pv = oracle.kv_cache_write(wv.pool, wv.k_new, wv.v_new, wv.slot_mapping)
    ref_ov, _ = oracle.paged_attention(wv.q, ref_pv, wv.block_table, wv.cu_seqlens, wv.seq_lens,
                                       wv.scale)
    devv = gu.DeviceStep(wv)
    devv.write()
    outv = torch.full(tuple(devv.q.shape), float("nan"), dtype=torch.float32, device="cuda")
    pkv.paged_attention_varlen(devv.q, devv.pool, devv.table, devv.cu, devv.lens, 1,
                               wv.max_seq_len, out=outv, scale=wv.scale, dev_status=devv.status)
    assert devv.dev_status() & gu.pkv.DEV_BAD_LENGTHS
    assert np.max(np.abs(outv.cpu().numpy()[0] - ref_ov[0])) <= gu.ATOL  # request 0 untouched
    # a slot outside the pool
    dev.status.zero_()
    slots = w.slot_mapping.copy()
    slots[0] = w.num_blocks * w.block_size + 3
    pkv.kv_cache_write(dev.pool, dev.k_new, dev.v_new, gu.i32_tensor(slots),
                       dev_status=dev.status)
    assert dev.dev_status() & gu.pkv.DEV_BAD_SLOT


@pytest.mark.parametrize("partition_size", [16, 48, 128, 1024])
def test_partition_sizes_with_verification_requests(oracle, partition_size):
    """Split-KV partition sizes on a batch that mixes one-query requests
    (split) with several-query verification requests (one partition each,
    the causal limit per row)."""
    w = wl.build("mqparts", [100, 257, 1030, 2049, 3001, 40, 777], [2, 8, 5, 3, 7, 4, 1],
                 32, 8, 128, seed=217)
    _run_and_check(oracle, w, partition_size)


def test_short_request_without_decode_grid_is_flagged(oracle):
    """num_tokens = 200 rows of q with max_query_len 100 over two requests
    shows that no request can be short, so no decode grid is launched;
    cu_seqlens_q disagrees (request 1 has 4 queries): that request is flagged,
    request 0 is still exact."""
    w = wl.build("nodec", [300, 40], [100, 4], 32, 8, 128, seed=216)
    ref_pool = oracle.kv_cache_write(w.pool, w.k_new, w.v_new, w.slot_mapping)
    ref_o, ref_l = oracle.paged_attention(w.q, ref_pool, w.block_table, w.cu_seqlens,
                                          w.seq_lens, w.scale)
    dev = gu.DeviceStep(w)
    dev.write()
    q = torch.zeros((200,) + tuple(dev.q.shape[1:]), dtype=dev.q.dtype, device="cuda")
    q[:104] = dev.q
    out = torch.full(tuple(q.shape), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full(tuple(q.shape[:2]), float("nan"), dtype=torch.float32, device="cuda")
    pkv.paged_attention_varlen(q, dev.pool, dev.table, dev.cu, dev.lens, 100, w.max_seq_len,
                               out=out, out_lse=lse, scale=w.scale, dev_status=dev.status)
    assert dev.dev_status() & gu.pkv.DEV_BAD_LENGTHS
    gu.compare(out[:100], lse[:100], ref_o[:100], ref_l[:100])


def test_debug_checks_name_the_bad_entry(oracle, monkeypatch):
    """With PKV_DEBUG_CHECKS=1 the binding checks the tables on the host
    before each call: a bad block id raises, naming the entry, before any
    launch; valid tables pass and the call runs as usual."""
    w = wl.build("dbg", [40, 300, 50], [1, 1, 20], 32, 8, 128, seed=302)
    dev = gu.DeviceStep(w)
    monkeypatch.setenv("PKV_DEBUG_CHECKS", "1")
    dev.write()
    bad = w.block_table.copy()
    bad[1, 3] = w.num_blocks + 5
    with pytest.raises(ValueError, match=r"block_table\[1\]\[3\]"):
        dev.attend(table=gu.i32_tensor(bad))
    assert dev.dev_status() == 0   # nothing ran
    _run_and_check(oracle, w)


@pytest.mark.parametrize("P,T,H,D", [(1, 3, 4, 128), (5, 7, 32, 128), (64, 2, 8, 64),
                                     (3, 4, 2, 256), (2, 1, 1, 4)])
def test_public_lse_merge(oracle, P, T, H, D):
    rng = np.random.default_rng(214 + P + D)
    po = rng.standard_normal((P, T, H, D)).astype(np.float32)
    pl = (rng.standard_normal((P, T, H)) * 3).astype(np.float32)
    if P > 1:
        pl[0, 0] = -np.inf          # an empty partition
        po[0, 0] = np.nan           # ... whose output must never enter a sum
        pl[:, -1, -1] = -np.inf     # a row with no keys at all
    ref_o, ref_l = oracle.lse_merge(po.astype(np.float64), pl.astype(np.float64))
    lse = torch.empty((T, H), dtype=torch.float32, device="cuda")
    out, _ = pkv.lse_merge(torch.from_numpy(po).cuda(), torch.from_numpy(pl).cuda(), out_lse=lse)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    l = lse.cpu().numpy()
    assert np.all(np.isfinite(o))
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(l), fin)
    assert np.max(np.abs(o - ref_o)) <= 1e-5
    if fin.any():
        assert np.max(np.abs(l[fin] - ref_l[fin])) <= 1e-5


def test_v_beyond_fp16_range_is_flagged(oracle):
    """The prefill kernel computes P.V in fp16 (exact for |v| < 65536, bf16
    values converted losslessly); a V value beyond that range in a context it
    reads sets PKV_DEV_V_RANGE. An ordinary workload never sets it, and a V
    value at the edge of the range (65280, the largest bf16 below 2^16) does
    not either."""
    w = wl.build("vrange", [500, 700], [1, 200], 32, 8, 128, seed=77)
    for value, flagged in ((0x477F, False), (0x47C3, True)):   # 65280, 100000
        pool = w.pool.copy()
        blk = int(w.block_table[1, 3])          # a context block of the prefill request
        pool[1, blk, 5, 2, 17] = value          # V half, token 5, KV head 2, element 17
        wv = wl.Workload(**{**w.__dict__, "pool": pool})
        dev = gu.DeviceStep(wv)
        dev.write()
        dev.attend()
        st = dev.dev_status()
        assert bool(st & pkv.DEV_V_RANGE) == flagged, st
        assert st & ~pkv.DEV_V_RANGE == 0
