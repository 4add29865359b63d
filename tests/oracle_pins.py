"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with what the pages or the mathematics fix:

* values the pages print (KV sizing worked example, GQA cache fraction,
  block-table examples) from ``tests/golden``;
* brute force: contiguous attention through ``torch``'s scaled-dot-product
  attention in fp64 with an explicit bottom-right causal mask, and a pure
  Python triple loop on a tiny case;
* closed forms (two keys whose scores differ by ln 3 give weights 1/4, 3/4;
  one key returns its V row; equal keys give the mean of V);
* invariants (block permutation, copy-on-write aliasing, GQA = MHA with
  repeated KV heads, decode = last prefill row, chunked = unchunked prefill,
  split-KV partitions merged by log-sum-exp = unsplit).

The same functions run against deliberately broken copies of the oracle in
``test_oracle_mutants.py``: every planted mistake must trip at least one pin.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

from paged_kv_cache_varlen_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name: str) -> dict:
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _f64(bits: np.ndarray) -> np.ndarray:
    return wl.bf16_bits_to_f32(bits).astype(np.float64)


def _written_pool(oracle, w: wl.Workload) -> np.ndarray:
    return oracle.kv_cache_write(w.pool, w.k_new, w.v_new, w.slot_mapping)


def _attend(oracle, w: wl.Workload, pool=None, **kw):
    pool = _written_pool(oracle, w) if pool is None else pool
    return oracle.paged_attention(w.q, pool, w.block_table, w.cu_seqlens, w.seq_lens, w.scale,
                                  **kw)


def _contiguous_kv(w: wl.Workload, i: int):
    """K, V [L, Hkv, D] of request i: cached history read from the (unwritten)
    pool by walking the block table, then the step's new rows taken straight
    from k_new / v_new. Independent of the oracle's KV write."""
    L, ql = int(w.seq_lens[i]), int(w.query_lens[i])
    BS = w.block_size
    ks, vs = [], []
    for p in range(L - ql):
        blk = int(w.block_table[i, p // BS])
        ks.append(w.pool[0, blk, p % BS])
        vs.append(w.pool[1, blk, p % BS])
    t0 = int(w.cu_seqlens[i])
    for j in range(ql):
        ks.append(w.k_new[t0 + j])
        vs.append(w.v_new[t0 + j])
    shape = (0, w.num_kv_heads, w.head_dim)
    k = np.stack(ks) if ks else np.zeros(shape, np.uint16)
    v = np.stack(vs) if vs else np.zeros(shape, np.uint16)
    return _f64(k), _f64(v)


def sdpa_reference(w: wl.Workload):
    """Contiguous attention per request via torch SDPA (fp64, explicit mask)."""
    import torch
    import torch.nn.functional as F

    T, H, D = w.q.shape
    G = w.num_heads // w.num_kv_heads
    out = np.zeros((T, H, D))
    lse = np.zeros((T, H))
    for i in range(w.num_seqs):
        L, ql = int(w.seq_lens[i]), int(w.query_lens[i])
        if ql == 0:
            continue
        t0 = int(w.cu_seqlens[i])
        k, v = _contiguous_kv(w, i)
        qi = torch.from_numpy(_f64(w.q[t0:t0 + ql])).permute(1, 0, 2)[None]          # 1,H,q,D
        ki = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]   # 1,H,L,D
        vi = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
        rows = torch.arange(ql)[:, None]
        cols = torch.arange(L)[None, :]
        mask = cols <= (L - ql) + rows                                                # bottom-right
        o = F.scaled_dot_product_attention(qi, ki, vi, attn_mask=mask, scale=w.scale)
        s = (qi @ ki.transpose(-1, -2)) * w.scale
        s = s.masked_fill(~mask, float("-inf"))
        out[t0:t0 + ql] = o[0].permute(1, 0, 2).numpy()
        lse[t0:t0 + ql] = torch.logsumexp(s, dim=-1)[0].permute(1, 0).numpy()
    return out, lse


SDPA_CASES = [
    # (seq_lens, query_lens, H, Hkv, D, BS, seed)
    ([1, 5, 16, 17, 40], [1, 1, 1, 1, 1], 4, 2, 16, 4, 11),     # decode, GQA 2
    ([9, 30, 3], [1, 7, 3], 6, 3, 8, 4, 12),                    # decode + chunk + full prefill
    ([33, 2], [2, 2], 4, 1, 32, 16, 13),                        # MQA, q = L
    ([20, 7, 12], [4, 1, 12], 2, 2, 8, 16, 14),                 # MHA
    ([1, 7, 16, 33], [1, 1, 1, 1], 4, 2, 64, 16, 1),            # the 4-request decode shape
]


def pin_sizing_worked_example(oracle):
    g = _golden("kv_cache_sizing.json")
    f = g["formula_factors"]
    heads, hd = g["llama2_7b_heads"], g["llama2_7b_head_dim"]
    assert heads * hd == f["hidden_size"]
    total = oracle.kv_cache_bytes(f["batch_size"], f["sequence_length"], f["num_layers"], heads,
                                  hd, f["bytes_per_element"])
    product = 1
    for v in f.values():
        product *= v
    assert total == product == 2 ** 31
    assert abs(total / 2 ** 30 - g["printed_result_gb_approx"]) < 1e-9
    per_token = oracle.kv_bytes_per_token(f["num_layers"], heads, hd, f["bytes_per_element"])
    assert per_token == 2 * f["num_layers"] * f["hidden_size"] * f["bytes_per_element"]


def pin_gqa_cache_fraction(oracle):
    g = _golden("kv_cache_sizing.json")
    gqa = oracle.kv_bytes_per_token(32, g["llama3_8b_kv_heads"], 128, 2)
    mha = oracle.kv_bytes_per_token(32, g["llama3_8b_q_heads"], 128, 2)
    assert gqa / mha == g["gqa_cache_fraction"]
    assert oracle.kv_bytes_per_token(1, 8, 128, 2) == 4096          # one layer, bf16
    assert gqa == 128 * 1024                                         # 32 layers


def pin_kv_write_closed_form(oracle):
    rng = np.random.default_rng(7)
    NB, BS, Hkv, D, T = 9, 4, 3, 8, 14
    pool = rng.integers(0, 2 ** 16, size=(2, NB, BS, Hkv, D), dtype=np.uint16)
    slots = rng.permutation(NB * BS)[:T].astype(np.int32)
    slots[[2, 9]] = -1
    k = rng.integers(0, 2 ** 16, size=(T, Hkv, D), dtype=np.uint16)
    v = rng.integers(0, 2 ** 16, size=(T, Hkv, D), dtype=np.uint16)
    new = oracle.kv_cache_write(pool, k, v, slots)
    flat_old = pool.reshape(2, NB * BS, Hkv, D)
    flat_new = new.reshape(2, NB * BS, Hkv, D)
    written = np.zeros(NB * BS, bool)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        written[s] = True
        assert np.array_equal(flat_new[0, s], k[t]) and np.array_equal(flat_new[1, s], v[t])
    assert np.array_equal(flat_new[:, ~written], flat_old[:, ~written])


def pin_kv_write_page_table(oracle):
    """Tokens 0..47 of a request whose table is the page's 57 -> 1024 -> 233."""
    table = _golden("block_tables.json")["logical_to_physical_example"]
    NB, BS, Hkv, D = 1100, 16, 1, 8
    pool = np.zeros((2, NB, BS, Hkv, D), np.uint16)
    pos = np.arange(48)
    slots = np.array([table[p // BS] * BS + p % BS for p in pos], np.int32)
    k = (np.arange(48, dtype=np.uint16)[:, None, None] + 1) * np.ones((1, Hkv, D), np.uint16)
    v = k + np.uint16(1000)
    new = oracle.kv_cache_write(pool, k, v, slots)
    for p in pos:
        assert np.all(new[0, table[p // BS], p % BS] == p + 1)
        assert np.all(new[1, table[p // BS], p % BS] == p + 1001)
    assert int((new != 0).sum()) == 2 * 48 * Hkv * D


def pin_attention_sdpa(oracle):
    for L, ql, H, Hkv, D, BS, seed in SDPA_CASES:
        w = wl.build("sdpa", L, ql, H, Hkv, D, BS, seed=seed, pool_factor=2.0)
        out, lse = _attend(oracle, w)
        ref_out, ref_lse = sdpa_reference(w)
        assert np.all(np.isfinite(out))
        np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def pin_attention_python_bruteforce(oracle):
    w = wl.build("py", [3, 4], [1, 2], 2, 1, 4, 2, seed=21)
    out, lse = _attend(oracle, w)
    G = w.num_heads // w.num_kv_heads
    for i in range(w.num_seqs):
        L, ql = int(w.seq_lens[i]), int(w.query_lens[i])
        k, v = _contiguous_kv(w, i)
        for j in range(ql):
            t = int(w.cu_seqlens[i]) + j
            for h in range(w.num_heads):
                qv = [float(x) for x in _f64(w.q[t, h])]
                scores = []
                for p in range(L - ql + j + 1):
                    scores.append(w.scale * sum(qv[d] * k[p, h // G, d] for d in range(w.head_dim)))
                z = sum(math.exp(s) for s in scores)
                for d in range(w.head_dim):
                    ref = sum(math.exp(s) / z * v[p, h // G, d] for p, s in enumerate(scores))
                    assert abs(out[t, h, d] - ref) < 1e-12
                assert abs(lse[t, h] - math.log(z)) < 1e-12


def _single_request(q_rows, k_rows, v_rows, scale, BS=4, query_len=1, table=None, NB=None):
    """A one-request workload with explicit bf16-exact float contents."""
    q_rows = np.asarray(q_rows, np.float32)
    k_rows = np.asarray(k_rows, np.float32)
    v_rows = np.asarray(v_rows, np.float32)
    L, D = k_rows.shape
    nblk = -(-L // BS)
    table = list(range(nblk)) if table is None else table
    NB = max(table) + 1 if NB is None else NB
    pool = np.full((2, NB, BS, 1, D), wl.BF16_NAN, np.uint16)
    for p in range(L):
        pool[0, table[p // BS], p % BS, 0] = wl.to_bf16_bits(k_rows[p])
        pool[1, table[p // BS], p % BS, 0] = wl.to_bf16_bits(v_rows[p])
    bt = np.array([table], np.int32)
    return (wl.to_bf16_bits(q_rows.reshape(query_len, 1, D)), pool, bt,
            np.array([0, query_len], np.int32), np.array([L], np.int32), scale)


def pin_two_key_closed_form(oracle):
    """Scores 0 and ln 3 give softmax weights 1/4 and 3/4."""
    a = 2.0
    args = _single_request([[1, 0]], [[0, 0], [a, 0]], [[4, -8], [12, 16]], math.log(3) / a)
    out, lse = oracle.paged_attention(*args)
    np.testing.assert_allclose(out[0, 0], [0.25 * 4 + 0.75 * 12, 0.25 * -8 + 0.75 * 16],
                               rtol=0, atol=1e-12)
    assert abs(lse[0, 0] - math.log(4.0)) < 1e-12


def pin_length_one_returns_v(oracle):
    w = wl.build("l1", [1, 1, 1], [1, 1, 1], 4, 2, 16, 4, seed=31)
    out, lse = _attend(oracle, w)
    G = w.num_heads // w.num_kv_heads
    for t in range(3):
        for h in range(4):
            assert np.array_equal(out[t, h], _f64(w.v_new[t, h // G]))
            s = w.scale * float(np.dot(_f64(w.q[t, h]), _f64(w.k_new[t, h // G])))
            assert abs(lse[t, h] - s) < 1e-12


def pin_probs_sum_to_one(oracle):
    w = wl.build("p", [40, 9], [3, 1], 4, 2, 8, 4, seed=41)
    pool = _written_pool(oracle, w)
    for t in range(w.num_tokens):
        for h in range(w.num_heads):
            p = oracle.attention_probs(w.q, pool, w.block_table, w.cu_seqlens, w.seq_lens,
                                       w.scale, t, h)
            i = int(np.searchsorted(w.cu_seqlens, t, side="right") - 1)
            j = t - int(w.cu_seqlens[i])
            assert p.shape[0] == int(w.seq_lens[i]) - int(w.query_lens[i]) + j + 1
            assert abs(p.sum() - 1.0) < 1e-12 and np.all(p > 0)


def pin_constant_keys_and_values(oracle):
    rng = np.random.default_rng(51)
    L, D = 11, 8
    vals = wl.bf16_bits_to_f32(wl.to_bf16_bits(rng.standard_normal((L, D), dtype=np.float32)))
    krow = wl.bf16_bits_to_f32(wl.to_bf16_bits(rng.standard_normal(D, dtype=np.float32)))
    qrow = wl.bf16_bits_to_f32(wl.to_bf16_bits(rng.standard_normal((1, D), dtype=np.float32)))
    out, _ = oracle.paged_attention(*_single_request(qrow, np.tile(krow, (L, 1)), vals, 0.3))
    np.testing.assert_allclose(out[0, 0], vals.astype(np.float64).mean(axis=0), rtol=0, atol=1e-12)
    keys = wl.bf16_bits_to_f32(wl.to_bf16_bits(rng.standard_normal((L, D), dtype=np.float32)))
    out, _ = oracle.paged_attention(*_single_request(qrow, keys, np.tile(vals[3], (L, 1)), 0.3))
    np.testing.assert_allclose(out[0, 0], vals[3].astype(np.float64), rtol=0, atol=1e-12)


def pin_block_permutation_invariance(oracle):
    w = wl.build("perm", [23, 40, 5], [1, 6, 5], 4, 2, 8, 4, seed=61, pool_factor=1.5)
    pool = _written_pool(oracle, w)
    out, lse = _attend(oracle, w, pool=pool)
    perm = np.random.default_rng(62).permutation(w.num_blocks)     # new id of old block b
    pool2 = np.empty_like(pool)
    pool2[:, perm] = pool
    bt2 = np.where(w.block_table >= 0, perm[np.maximum(w.block_table, 0)], -1).astype(np.int32)
    out2, lse2 = oracle.paged_attention(w.q, pool2, bt2, w.cu_seqlens, w.seq_lens, w.scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def pin_cow_aliasing_page_fixture(oracle):
    """Requests A = [7, 2] and B = [7, 6, 4] share physical block 7; giving B a
    private copy of that block must not change anything."""
    g = _golden("block_tables.json")
    a_tab, b_tab = g["cow_request_a"], g["cow_request_b"]
    BS, Hkv, H, D, NB = 16, 2, 4, 16, 12
    rng = np.random.default_rng(71)
    pool = wl.to_bf16_bits(rng.standard_normal((2, NB, BS, Hkv, D), dtype=np.float32))
    seq_lens = np.array([2 * BS, 3 * BS - 5], np.int32)
    cu = np.array([0, 1, 2], np.int32)
    q = wl.to_bf16_bits(rng.standard_normal((2, H, D), dtype=np.float32))
    bt = np.array([a_tab + [-1], b_tab], np.int32)
    out, lse = oracle.paged_attention(q, pool, bt, cu, seq_lens, 0.25)
    private = 9
    assert private not in a_tab + b_tab
    pool2 = pool.copy()
    pool2[:, private] = pool[:, g["shared_physical_block"]]
    bt2 = np.array([a_tab + [-1], [private] + b_tab[1:]], np.int32)
    out2, lse2 = oracle.paged_attention(q, pool2, bt2, cu, seq_lens, 0.25)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)
    # and the sharing is real: dropping the shared block changes request A
    pool3 = pool.copy()
    pool3[:, 7] = pool[:, 11]
    out3, _ = oracle.paged_attention(q, pool3, bt, cu, seq_lens, 0.25)
    assert not np.allclose(out3[0], out[0]) and not np.allclose(out3[1], out[1])


def pin_gqa_equals_repeated_mha(oracle):
    """Consecutive query heads h share KV head h // G; repeating every KV head
    G times (an MHA pool) gives the same result."""
    w = wl.build("gqa", [30, 12], [2, 1], 8, 2, 8, 4, seed=81)
    pool = _written_pool(oracle, w)
    out, lse = _attend(oracle, w, pool=pool)
    G = w.num_heads // w.num_kv_heads
    mha_pool = np.repeat(pool, G, axis=3)
    out2, lse2 = oracle.paged_attention(w.q, mha_pool, w.block_table, w.cu_seqlens, w.seq_lens,
                                        w.scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def pin_decode_equals_last_prefill_row(oracle):
    """Reusing cached K/V (decode, q = 1 at position L - 1) gives the last row
    of a prefill of all L tokens."""
    L = 37
    w = wl.build("pre", [L], [L], 4, 2, 8, 4, seed=91)
    pool = _written_pool(oracle, w)
    out, lse = _attend(oracle, w, pool=pool)
    cu = np.array([0, 1], np.int32)
    dec_out, dec_lse = oracle.paged_attention(w.q[L - 1:L], pool, w.block_table, cu,
                                              np.array([L], np.int32), w.scale)
    assert np.array_equal(dec_out[0], out[L - 1]) and np.array_equal(dec_lse[0], lse[L - 1])


def pin_chunked_equals_unchunked(oracle):
    L = 45
    w = wl.build("chunk", [L], [L], 4, 2, 8, 4, seed=101)
    pool = _written_pool(oracle, w)
    full, full_lse = _attend(oracle, w, pool=pool)
    for start, stop in [(0, 13), (13, 30), (30, 45)]:
        cu = np.array([0, stop - start], np.int32)
        o, l = oracle.paged_attention(w.q[start:stop], pool, w.block_table, cu,
                                      np.array([stop], np.int32), w.scale)
        assert np.array_equal(o, full[start:stop]) and np.array_equal(l, full_lse[start:stop])


def pin_merge_partitions_equal_full(oracle):
    w = wl.build("split", [1200, 700, 40], [1, 3, 1], 4, 2, 16, 16, seed=111)
    pool = _written_pool(oracle, w)
    full, full_lse = _attend(oracle, w, pool=pool)
    for size in (512, 256, 48):
        parts = [oracle.paged_attention(w.q, pool, w.block_table, w.cu_seqlens, w.seq_lens,
                                        w.scale, key_begin=b, key_end=b + size)
                 for b in range(0, 1200, size)]
        po = np.stack([p[0] for p in parts])
        pl = np.stack([p[1] for p in parts])
        out, lse = oracle.lse_merge(po, pl)
        np.testing.assert_allclose(out, full, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, full_lse, rtol=0, atol=1e-12)


def pin_cascade_prefix_plus_tail_equals_full(oracle):
    """Decode requests sharing a copy-on-write prefix: attention over the
    prefix alone (its blocks as their own table) merged by lse with attention
    over each private tail (the table shifted past the prefix) equals the
    attention over the whole context."""
    P, BS = 32, 8
    w = wl.build("cascade", [40, 33, 61, 45], [1, 1, 1, 1], 4, 2, 8, BS, seed=131,
                 shared_prefix=[([0, 1, 2], P)])
    pool = _written_pool(oracle, w)
    full, full_lse = _attend(oracle, w, pool=pool)
    members = [0, 1, 2]
    cu1 = np.arange(len(members) + 1, dtype=np.int32)
    ptable = np.repeat(w.block_table[:1, :P // BS], len(members), axis=0)
    po, pl = oracle.paged_attention(w.q[members], pool, ptable, cu1,
                                    np.full(len(members), P, np.int32), w.scale)
    ttable = np.ascontiguousarray(w.block_table[members, P // BS:])
    to, tl = oracle.paged_attention(w.q[members], pool, ttable, cu1,
                                    (w.seq_lens[members] - P).astype(np.int32), w.scale)
    out, lse = oracle.lse_merge(np.stack([po, to]), np.stack([pl, tl]))
    np.testing.assert_allclose(out, full[members], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, full_lse[members], rtol=0, atol=1e-12)
    # the prefix blocks really are shared by the group's tables
    assert (w.block_table[members, :P // BS] == w.block_table[0, :P // BS]).all()


def pin_merge_single_and_empty_partitions(oracle):
    rng = np.random.default_rng(121)
    o = rng.standard_normal((1, 5, 3, 8))
    l = rng.standard_normal((1, 5, 3))
    out, lse = oracle.lse_merge(o, l)
    assert np.array_equal(out, o[0]) and np.array_equal(lse, l[0])
    junk = np.full_like(o, np.nan)
    empty = np.full_like(l, -np.inf)
    out2, lse2 = oracle.lse_merge(np.concatenate([junk, o, junk]),
                                  np.concatenate([empty, l, empty]))
    np.testing.assert_allclose(out2, o[0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse2, l[0], rtol=0, atol=1e-15)
    out3, lse3 = oracle.lse_merge(junk, empty)
    assert np.all(out3 == 0) and np.all(lse3 == -np.inf)
    # two equal partials: same output, lse + ln 2
    out4, lse4 = oracle.lse_merge(np.concatenate([o, o]), np.concatenate([l, l]))
    np.testing.assert_allclose(out4, o[0], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse4, l[0] + math.log(2.0), rtol=0, atol=1e-14)


def pin_rejects_bad_inputs(oracle):
    import oracle as oracle_pkg

    w = wl.build("bad", [20], [1], 4, 2, 8, 4, seed=131)
    pool = _written_pool(oracle, w)
    bad = w.block_table.copy()
    bad[0, 2] = w.num_blocks
    for kwargs in ({"block_table": bad},
                   {"seq_lens": np.array([0], np.int32)},
                   {"cu_seqlens": np.array([0, 2], np.int32)}):
        args = dict(q=w.q, pool=pool, block_table=w.block_table, cu_seqlens=w.cu_seqlens,
                    seq_lens=w.seq_lens, scale=w.scale)
        args.update(kwargs)
        try:
            oracle.paged_attention(**args)
        except oracle_pkg.OracleError:
            continue
        raise AssertionError(f"oracle accepted bad input {list(kwargs)}")
    try:
        oracle.kv_cache_write(w.pool, w.k_new, w.v_new, np.array([w.num_blocks * 4], np.int32))
    except oracle_pkg.OracleError:
        pass
    else:
        raise AssertionError("oracle accepted an out-of-range slot")


ALL_PINS = [
    pin_cascade_prefix_plus_tail_equals_full,
    pin_sizing_worked_example,
    pin_gqa_cache_fraction,
    pin_kv_write_closed_form,
    pin_kv_write_page_table,
    pin_attention_sdpa,
    pin_attention_python_bruteforce,
    pin_two_key_closed_form,
    pin_length_one_returns_v,
    pin_probs_sum_to_one,
    pin_constant_keys_and_values,
    pin_block_permutation_invariance,
    pin_cow_aliasing_page_fixture,
    pin_gqa_equals_repeated_mha,
    pin_decode_equals_last_prefill_row,
    pin_chunked_equals_unchunked,
    pin_merge_partitions_equal_full,
    pin_merge_single_and_empty_partitions,
    pin_rejects_bad_inputs,
]
