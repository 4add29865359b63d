"""bench.py's multi-rank host logic on CPU: two gloo ranks (no GPU).

With torchrun every rank runs an independent replica; the job's time is the
slowest rank's and its throughput counts the bytes of every rank. These tests
run that reduction over a real two-process gloo group, check that the ranks
get different batches of the same shape, and that the reference arm leaves
rank 1 without doing any work.
"""
import json
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

WORLD = 2


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, out_dir):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench as b

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(WORLD), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        mine = {"total_ms": 100.0 + 25.0 * rank, "e2e_ms": 300.0 - 40.0 * rank,
                "attn_avg_ms": 0.5 + 0.25 * rank}
        slowest = b.max_over_ranks(mine, dist, "cpu")
        w = b.rank_workload("tiny", rank)
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"slowest": slowest, "world": b.dist_info()[0],
                       "seq_lens": w.seq_lens.tolist(), "q_sum": int(w.q.astype(np.int64).sum()),
                       "q_shape": list(w.q.shape), "kv_bytes": w.kv_bytes()}, f)
    finally:
        dist.destroy_process_group()


@pytest.fixture(scope="module")
def two_ranks(tmp_path_factory):
    out_dir = str(tmp_path_factory.mktemp("ranks"))
    mp.start_processes(_rank_main, args=(_free_port(), out_dir), nprocs=WORLD, join=True,
                       start_method="spawn")
    res = []
    for r in range(WORLD):
        with open(os.path.join(out_dir, f"rank{r}.json")) as f:
            res.append(json.load(f))
    return res


def test_every_rank_sees_the_slowest_time(two_ranks):
    want = {"total_ms": 125.0, "e2e_ms": 300.0, "attn_avg_ms": 0.75}
    for r in two_ranks:
        assert r["world"] == WORLD
        assert r["slowest"] == want


def test_replicas_get_independent_batches_of_one_shape(two_ranks):
    a, b = two_ranks
    assert a["q_shape"] == b["q_shape"] and a["seq_lens"] == b["seq_lens"]
    assert a["kv_bytes"] == b["kv_bytes"]
    assert a["q_sum"] != b["q_sum"]


def test_job_throughput_counts_every_rank():
    # 2 ranks x 1e9 bytes each in 0.5 ms per step -> 4000 GB/s for the job
    assert bench.job_throughput(2, 10**9, 0.5) == pytest.approx(4000.0)
    assert bench.job_throughput(1, 10**9, 0.5) == pytest.approx(2000.0)


def test_no_group_means_local_values():
    v = {"total_ms": 3.0}
    assert bench.max_over_ranks(v) == v


def test_reference_arm_rank1_does_no_work(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
    assert bench.main() == 0
    assert capsys.readouterr().out == ""


def test_split_parts_follows_the_library():
    """bench.py counts the merge grid from its own copy of the partition
    rule; the library's workspace size (partials for every partition) pins
    that copy: partials exist exactly when the count is above 1, and their
    size is the count's."""
    from paged_kv_cache_varlen_gb300 import binding
    lib = binding.load_library()
    B, H, D = 8, 32, 128
    up = lambda x: -(-x // 256) * 256
    for L in (1, 16, 1000, 1024, 1025, 4096, 4097, 32768, 32769, 131072, 200000):
        for ps in (-1, 0, 16, 512, 2048):
            n = bench.split_parts(L, ps)
            ws = lib.pkv_attention_workspace_size(B, B, H, 8, D, L, ps)
            rows = B * n * H
            want = 256 if n == 1 else up(rows * D * 4) + up(rows * 4) + 256
            assert ws == want, (L, ps, n, ws, want)


def test_packed_inputs_round_trip():
    """The end-to-end step copies all of its inputs in one packed buffer;
    the views bench.py hands to the kernels must hold exactly the inputs,
    at 256-byte aligned offsets (the kernels need 16-byte alignment)."""
    import torch
    rng = np.random.default_rng(3)
    host = {
        "q": torch.from_numpy(rng.integers(-2**15, 2**15, size=(5, 4, 64), dtype=np.int16)
                              ).view(torch.bfloat16),
        "slots": torch.from_numpy(rng.integers(0, 1000, size=7, dtype=np.int32)),
        "table": torch.from_numpy(rng.integers(0, 1000, size=(3, 9), dtype=np.int32)),
        "cu": torch.from_numpy(np.array([0, 2, 5, 7], dtype=np.int32)),
    }
    offs, total, buf = bench.pack_inputs(host)
    assert total % 256 == 0 and all(o % 256 == 0 for o, _ in offs.values())
    views = bench.unpack_views(buf.clone(), offs, host)
    for k, v in host.items():
        assert views[k].dtype == v.dtype and views[k].shape == v.shape
        assert torch.equal(views[k].view(torch.uint8), v.view(torch.uint8)), k
