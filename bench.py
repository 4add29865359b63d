#!/usr/bin/env python3
"""Benchmark of one paged-attention step on GB300.

A step is the whole hot path over one batch: the KV write of the step's new
K/V rows (slot_mapping) followed by varlen paged attention (decode kernel,
split-KV log-sum-exp merge, chunked-prefill kernel as the batch needs).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config llama3_8b_decode]

Prints ONE JSON line (rank 0). ``value`` is KV GB/s (algorithmic bytes: every
request reads its whole context once, 2*Hkv*D*2 bytes per token) over the
device-resident step time; ``e2e`` repeats the measurement with the step's
inputs copied from pinned host memory and the output copied back inside the
timed region. ``--impl reference`` times the fp64 CPU oracle on the host
cores instead (bounded sample of the same workload).

Multi-GPU (torchrun): every rank runs an independent replica on its own GPU
(requests are independent, so the path shards with no collective); timing is
the max over ranks, ``value`` the total bytes of all ranks over that time.
"""
from __future__ import annotations

import argparse
import gc
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="llama3_8b_decode")
    ap.add_argument("--partition-size", type=int, default=-1)
    ap.add_argument("--cascade", action="store_true",
                    help="prefix_cow only: read each shared prefix once per group "
                         "(pkv_cascade_decode) instead of once per request")
    ap.add_argument("--separate-write", action="store_true",
                    help="time each step as pkv_kv_cache_write then the attention call, "
                         "instead of the combined pkv_paged_attention_varlen_append")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--extra", default=EXTRA_DEFAULT,
                    help="comma-separated workloads also timed device-resident in the same "
                         "run and reported under 'workloads' ('none' to skip); a name "
                         "ending in '+cascade' runs it as the cascade call")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target length of the oracle CPU-baseline sample")
    ap.add_argument("--ref-seconds", type=float, default=150.0,
                    help="target length of the whole --impl reference run")
    return ap.parse_args()


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense bf16 TFLOP/s: the measured burst figure, else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def split_parts(max_seq_len: int, partition_size: int) -> int:
    """Split-KV partitions per request, as the library resolves them: 1024
    tokens doubled until at most 32 (automatic), none (0) or the given size."""
    length = max(int(max_seq_len), 1)
    if partition_size == 0:
        return 1
    s = 1024 if partition_size < 0 else partition_size
    while partition_size < 0 and -(-length // s) > 32:
        s *= 2
    return max(1, -(-length // s))


def attention_launches(w, partition_size: int, ci) -> int:
    """Kernels one attention call launches: the decode grid and, when
    requests split, its merge grid; before them, for a decode-only batch with
    several-query requests and at most 256 requests, the one-CTA kernel that
    orders the requests longest first; with requests longer than the decode
    kernel takes, the prefill grid first, and the decode grids behind it only
    when some request may be short (num_seqs * max_query_len - num_tokens >=
    max_query_len - max(1, 32 / G)). The cascade call: the prefix pass, the
    tail decode (and its merge grid when tails split) and the final merge;
    the tail decode alone when there is no prefix."""
    if ci is not None:
        tail = 1 + (1 if split_parts(ci["max_tail_len"], -1) > 1 else 0)
        prefixes = len(ci["prefix_lens"]) > 0 and ci["max_prefix_len"] > 0
        return tail + (2 if prefixes else 0)
    group = w.num_heads // w.num_kv_heads
    dmq = max(1, 32 // group)
    decode = 1 + (1 if split_parts(w.max_seq_len, partition_size) > 1 else 0)
    if w.max_query_len <= dmq:
        # several-query batches of at most 256 requests: the order kernel first
        ordered = w.num_tokens > w.num_seqs and w.num_seqs <= 256
        return decode + (1 if ordered else 0)
    may_be_short = w.num_seqs * w.max_query_len - w.num_tokens >= w.max_query_len - dmq
    return 1 + (decode if may_be_short else 0)


def pack_inputs(tensors: dict, align: int = 256):
    """Lay contiguous tensors end to end in one byte buffer, each piece at an
    `align`-byte offset. Returns ({name: (offset, bytes)}, total bytes, the
    packed uint8 tensor)."""
    import torch

    offs, total = {}, 0
    for k, v in tensors.items():
        offs[k] = (total, v.numel() * v.element_size())
        total = -(-(total + offs[k][1]) // align) * align
    buf = torch.zeros(total, dtype=torch.uint8)
    for k, v in tensors.items():
        o, n = offs[k]
        buf[o:o + n].copy_(v.reshape(-1).view(torch.uint8))
    return offs, total, buf


def unpack_views(buf, offs: dict, like: dict) -> dict:
    """Views of a packed byte buffer with the dtypes and shapes of `like`."""
    return {k: buf[o:o + n].view(like[k].dtype).view(like[k].shape)
            for k, (o, n) in offs.items()}


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("decode_mma.cu", "common.cuh"):  # the decode and merge grids' sources
        with open(os.path.join(ROOT, "paged_kv_cache_varlen_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(config: str):
    """DRAM bytes per attention launch from the committed ncu summary, or
    None when the summary is missing or the kernels changed since."""
    path = os.path.join(ROOT, "profiles", f"decode_{config}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    m_val = re.search(r"traffic_bytes_per_attention_call:\s*([0-9]+)", text)
    if not m_hash or not m_val or m_hash.group(1) != kernel_source_hash():
        return None
    return int(m_val.group(1))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 50 ms while the
    timed work runs. The median SM clock is taken over the samples that saw
    the GPU busy (utilization >= 50 %), so idle gaps do not pull it down."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "utilization.gpu")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    @staticmethod
    def summarise(text: str) -> dict:
        sm, smax, busy, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in text.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                mhz, mx, util = float(parts[1]), float(parts[2]), float(parts[9])
            except ValueError:
                continue
            sm.append(mhz)
            smax.append(mx)
            if util >= 50.0:
                busy.append(mhz)
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        pick = busy if busy else sm
        return {"sm_mhz": statistics.median(pick) if pick else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "samples_under_load": len(busy)}

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "samples_under_load": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return self.summarise(out)


def l2_size(device=None) -> int:
    """L2 bytes of the GPU (both arms report the same figure on one box)."""
    try:
        import torch

        if torch.cuda.is_available():
            return int(torch.cuda.get_device_properties(device if device is not None else 0)
                       .L2_cache_size)
    except Exception:
        pass
    return 126 * 2**20


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


SEEDS = {"tiny": 1, "llama3_8b_decode": 2, "long_split_kv": 3, "prefix_cow": 4, "mixed_step": 5,
         "prefill_chunks": 5, "spec_verify": 6}


def rank_workload(config: str, rank: int, poison: bool = False):
    """The batch one rank processes: the workload's own seed on rank 0, a
    different seed per rank elsewhere (replicas see independent requests of
    the same shape)."""
    from paged_kv_cache_varlen_gb300 import workloads as wl

    return wl.CONFIGS[config](seed=SEEDS[config] + 1000 * rank, poison=poison)


def max_over_ranks(values: dict, dist=None, device="cpu") -> dict:
    """Per-key maximum over ranks of this rank's timings: the slowest rank
    sets the job's time. Without a process group the values come back as is."""
    if dist is None:
        return dict(values)
    import torch

    keys = sorted(values)
    t = torch.tensor([float(values[k]) for k in keys], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return dict(zip(keys, t.tolist()))


def job_throughput(world: int, bytes_per_rank: int, ms_per_step: float) -> float:
    """Whole-job GB/s: the bytes every rank processed in one step over the
    slowest rank's step time (weak scaling: each rank keeps its own batch)."""
    return world * bytes_per_rank / (ms_per_step * 1e-3) / 1e9


def pool_copies(unique_kv_bytes: int, l2_bytes: int) -> int:
    """Copies of the KV pool the timed loops rotate through so that no step
    finds the previous step's K/V in L2: one when a step reads more than
    twice the L2 size, else enough that the other copies hold over twice it."""
    if unique_kv_bytes >= 2 * l2_bytes:
        return 1
    return min(64, -(-2 * l2_bytes // max(unique_kv_bytes, 1)) + 1)


def workload_config(w, partition_size: int, world: int, copies: int = 1,
                    l2_bytes: int = 126 * 2**20) -> dict:
    unique = w.unique_kv_bytes() if "prefix_tokens" in w.meta else w.kv_bytes()
    if (copies - 1) * unique < 2 * l2_bytes and copies > 1:
        l2 = (f"L2-resident: the KV read per step is small enough that even {copies} "
              "rotated pool copies fit in L2")
    elif copies == 1:
        l2 = (f"inputs larger than L2 (KV read per step >= 2 x {l2_bytes >> 20} MB L2), "
              "no flush")
    else:
        l2 = (f"KV pool rotated over {copies} copies, step k on copy k mod {copies} "
              f"(the others hold > 2 x {l2_bytes >> 20} MB L2), no flush")
    return {"workload": w.name, "num_seqs": w.num_seqs, "num_heads": w.num_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
            "block_size": w.block_size, "max_seq_len": w.max_seq_len,
            "kv_bytes_per_step": w.kv_bytes(), "partition_size": partition_size,
            "l2": l2, "parallelism": f"replicas x{world}"}


def oracle_step(orc, w):
    """One oracle step of the workload: the KV write, then attention of every
    request (the whole hot path, in fp64 on the host cores)."""
    pool = orc.kv_cache_write(w.pool, w.k_new, w.v_new, w.slot_mapping)
    orc.paged_attention(w.q, pool, w.block_table, w.cu_seqlens, w.seq_lens, w.scale)


def oracle_step_seconds(w, budget_s: float, threads: int = 0):
    """Time the oracle on whole steps of the workload; repeat until about
    `budget_s` seconds of CPU time. Returns the median step time, the
    threads used (all cores of the affinity mask unless `threads` is given)
    and the number of steps."""
    import oracle as oracle_pkg

    orc = oracle_pkg.load()
    orc.set_num_threads(threads if threads > 0 else len(os.sched_getaffinity(0)))
    cores = orc.num_threads()
    times = []
    t_all = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        oracle_step(orc, w)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_all >= budget_s or len(times) >= 50:
            break
    return statistics.median(times), cores, len(times)


def work_units(w) -> np.ndarray:
    """Keys scanned per request (context length x query rows), a proxy for
    the oracle's time on it."""
    return w.seq_lens.astype(np.int64) * w.query_lens.astype(np.int64)


def oracle_sample(w, max_units: int = 4_000_000):
    """A bounded sample of the workload for the oracle: the whole batch when
    its work fits `max_units`, otherwise its first requests (at least one)."""
    from paged_kv_cache_varlen_gb300 import workloads as wl

    cum = np.cumsum(work_units(w))
    if cum[-1] <= max_units:
        return w, f"whole batch ({w.num_seqs} requests)"
    keep = max(1, min(int(np.searchsorted(cum, max_units, side="right")), w.num_seqs))
    sub = wl.build(w.name + "_sample", w.seq_lens[:keep], w.query_lens[:keep], w.num_heads,
                   w.num_kv_heads, w.head_dim, w.block_size, seed=w.seed, poison=False)
    return sub, f"first {keep} of {w.num_seqs} requests"


def run_reference(args):
    """The reference arm: the fp64 oracle, as it stands, on the host cores.
    W untimed and K timed steps, each over a bounded sample of the workload
    sized so that the whole run takes about --ref-seconds. Under torchrun only
    rank 0 runs it; the other ranks leave at once."""
    world, rank, _ = dist_info()
    if rank != 0:
        return 0
    import oracle as oracle_pkg

    orc = oracle_pkg.load()
    w = rank_workload(args.config, 0)
    K, W = max(1, args.steps), max(3, args.warmup)
    # size the sample from the time of the first request alone
    first, _ = oracle_sample(w, 1)
    t0 = time.perf_counter()
    oracle_step(orc, first)
    sec_per_unit = (time.perf_counter() - t0) / float(work_units(first).sum())
    per_step = args.ref_seconds / (K + W)
    sample, desc = oracle_sample(w, int(per_step / sec_per_unit))
    for _ in range(W):
        oracle_step(orc, sample)
    t0 = time.perf_counter()
    for _ in range(K):
        oracle_step(orc, sample)
    sec = (time.perf_counter() - t0) / K
    gbs = sample.kv_bytes() / sec / 1e9
    cores = orc.num_threads()
    line = {
        "impl": "reference", "metric": "paged decode attention KV GB/s", "value": gbs,
        "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": sec * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "seqs_per_s": sample.num_seqs / sec,
        "config": workload_config(w, args.partition_size, world,
                                  pool_copies(w.kv_bytes(), l2_size()), l2_size()),
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{desc} of the rank-0 batch, every step"},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


EXTRA_DEFAULT = "long_split_kv,spec_verify,mixed_step,prefill_chunks,prefix_cow+cascade"


class DeviceWorkload:
    """One rank's batch of a workload resident on its GPU: the packed per-step
    inputs (pinned on the host and on the device), the KV pool (rotated over
    copies when a step's KV read is smaller than twice the L2), the outputs
    and the workspace, and the calls of one step."""

    def __init__(self, w, dev, stream, partition_size: int, cascade: bool, l2_bytes: int):
        import torch

        from paged_kv_cache_varlen_gb300 import binding as pkv
        from paged_kv_cache_varlen_gb300 import workloads as wl

        self.w, self.dev, self.stream, self.pkv = w, dev, stream, pkv
        self.partition_size = partition_size
        self.separate_write = False
        T, H, D = w.q.shape

        def bf16(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)

        host = {"q": bf16(w.q), "k_new": bf16(w.k_new), "v_new": bf16(w.v_new),
                "slots": torch.from_numpy(w.slot_mapping)}
        self.ci = None
        if cascade:
            if "prefix_tokens" not in w.meta:
                raise SystemExit("--cascade needs a workload with shared prefixes (prefix_cow)")
            self.ci = wl.cascade_inputs(w, wl.prefix_groups(w))
            for k in ("group_starts", "prefix_lens", "prefix_tables", "tail_tables",
                      "tail_lens"):
                host[k] = torch.from_numpy(self.ci[k])
        else:
            host["table"] = torch.from_numpy(w.block_table)
            host["cu"] = torch.from_numpy(w.cu_seqlens)
            host["lens"] = torch.from_numpy(w.seq_lens)
        # every per-step input packed into one pinned host buffer, so that a
        # step's inputs travel in one copy
        self.host = host
        self.offs, self.total_in, buf = pack_inputs(host)
        self.host_buf = buf.pin_memory()
        self.d_buf, self.d = self.device_set()
        self.d_buf.copy_(self.host_buf)
        pool = bf16(w.pool).to(dev)
        unique = w.unique_kv_bytes() if "prefix_tokens" in w.meta else w.kv_bytes()
        self.n_pools = pool_copies(unique, l2_bytes)
        self.pools = [pool] + [pool.clone() for _ in range(self.n_pools - 1)]
        self.out = torch.empty((T, H, D), dtype=torch.float32, device=dev)
        self.lse = torch.empty((T, H), dtype=torch.float32, device=dev)
        if self.ci is not None:
            ci = self.ci
            ws_bytes = pkv.cascade_workspace_size(w.num_seqs, len(ci["prefix_lens"]),
                                                  ci["max_group_size"], ci["max_prefix_len"],
                                                  ci["max_tail_len"], H, w.num_kv_heads, D)
        else:
            ws_bytes = pkv.attention_workspace_size(w.num_seqs, T, H, w.num_kv_heads, D,
                                                    w.max_seq_len, partition_size)
        self.ws = torch.zeros(max(ws_bytes, 1), dtype=torch.uint8, device=dev)

    def device_set(self):
        import torch

        buf = torch.empty(self.total_in, dtype=torch.uint8, device=self.dev)
        return buf, unpack_views(buf, self.offs, self.host)

    def attend(self, dd=None, ev=None, res=None, k=0):
        w, pkv, ci = self.w, self.pkv, self.ci
        dd = self.d if dd is None else dd
        o, ls = (self.out, self.lse) if res is None else res
        pool = self.pools[k % self.n_pools]
        if ev is not None:
            ev[0].record(self.stream)
        if ci is not None:
            pkv.cascade_decode(dd["q"], pool, dd["group_starts"], dd["prefix_lens"],
                               dd["prefix_tables"], ci["max_group_size"], ci["max_prefix_len"],
                               dd["tail_tables"], dd["tail_lens"], ci["max_tail_len"], out=o,
                               out_lse=ls, scale=w.scale, workspace=self.ws, stream=self.stream)
        else:
            pkv.paged_attention_varlen(dd["q"], pool, dd["table"], dd["cu"], dd["lens"],
                                       w.max_query_len, w.max_seq_len, out=o, out_lse=ls,
                                       scale=w.scale, partition_size=self.partition_size,
                                       workspace=self.ws, stream=self.stream)
        if ev is not None:
            ev[1].record(self.stream)

    def step(self, dd=None, res=None, k=0):
        """One step: the KV write and the attention call. By default in one
        call (pkv_paged_attention_varlen_append); the cascade call, and every
        call with separate_write set, as the two calls one after the other."""
        dd = self.d if dd is None else dd
        pool = self.pools[k % self.n_pools]
        if self.ci is not None or self.separate_write:
            self.pkv.kv_cache_write(pool, dd["k_new"], dd["v_new"], dd["slots"],
                                    stream=self.stream)
            self.attend(dd, res=res, k=k)
            return
        w = self.w
        o, ls = (self.out, self.lse) if res is None else res
        self.pkv.paged_attention_varlen_append(
            dd["q"], pool, dd["k_new"], dd["v_new"], dd["slots"], dd["table"], dd["cu"],
            dd["lens"], w.max_query_len, w.max_seq_len, out=o, out_lse=ls, scale=w.scale,
            partition_size=self.partition_size, workspace=self.ws, stream=self.stream)

    def timed(self, fn, K: int) -> float:
        """ms of K calls of fn(k) back to back between one pair of events (an
        event recorded between two kernels would also stop the next one from
        launching early under programmatic dependent launch)."""
        import torch

        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(self.dev)
        # Hold the stream (a bounded sleep on the device, before the first
        # event) while the host enqueues the calls: ~150 us a call, at least
        # 0.2 ms and at most 20 ms. The region then measures the device's
        # time for the K calls, not the host's latency to issue them (a step
        # of two API calls takes the host about as long as the device).
        # The host must stay ahead of the device for the whole region: the
        # garbage collector is off inside it (a full collection can hold the
        # host for tens of ms while the device drains its queue).
        gc.collect()
        gc.disable()
        try:
            hold_us = min(20_000, max(200, 150 * K))
            with torch.cuda.stream(self.stream):
                torch.cuda._sleep(2_000 * hold_us)  # cycles at ~2 GHz
            a.record(self.stream)
            t0 = time.perf_counter()
            for k in range(K):
                fn(k)
            self.last_host_us = (time.perf_counter() - t0) * 1e6 / K
            b.record(self.stream)
            torch.cuda.synchronize(self.dev)
        finally:
            gc.enable()
        return a.elapsed_time(b)

    def launches_per_step(self) -> int:
        return 1 + attention_launches(self.w, self.partition_size, self.ci)


def roofline_and_prefill(w, attn_avg_ms: float, ci=None) -> tuple:
    """(roofline, prefill) objects of one workload's attention call: KV bytes
    over the call's time against the measured HBM peak (unique bytes for
    shared prefixes), and for batches with requests on the tensor-core
    prefill kernel their causal-exact TFLOP/s and the serial bound T*."""
    peak, peak_kind = hbm_peak()
    kv_bytes = w.kv_bytes()
    roof_bytes = w.unique_kv_bytes() if "prefix_tokens" in w.meta else kv_bytes
    achieved = roof_bytes / (attn_avg_ms * 1e-3) / 1e9
    roof = {"bound": "hbm",
            "kernel": ("cascade call (prefix pass + tail decode + merge)" if ci is not None
                       else "attention call (decode + split-KV merge"
                       + (" + prefill)" if w.max_query_len > max(1, 32 // (
                           w.num_heads // w.num_kv_heads)) else ")")),
            "bytes_per_call": roof_bytes, "achieved": achieved, "peak": peak,
            "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak}
    dmq = max(1, 32 // (w.num_heads // w.num_kv_heads))
    flops = w.attention_flops(dmq + 1)
    prefill = None
    if flops > 0:
        tpeak, tkind = tensor_peak()
        tflops = flops / (attn_avg_ms * 1e-3) / 1e12
        # serial bound of the whole call: every K/V byte at the HBM peak plus
        # the prefill FLOPs at the tensor peak
        t_star_us = 1e6 * (kv_bytes / (peak * 1e9) + flops / (tpeak * 1e12))
        prefill = {"flops_per_step": flops, "achieved_tflops": tflops, "peak_tflops": tpeak,
                   "peak_kind": tkind, "frac": tflops / tpeak, "t_star_us": t_star_us,
                   "t_star_frac": t_star_us / (attn_avg_ms * 1e3),
                   "time": "attention call" + (" (decode kernel included)"
                                               if (w.query_lens <= dmq).any() else "")}
    return roof, prefill


def run_ours(args):
    import torch

    from paged_kv_cache_varlen_gb300 import binding as pkv
    from paged_kv_cache_varlen_gb300 import build as pkv_build

    world, rank, local = dist_info()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    pkv_build.build()
    pkv.load_library()
    stream = torch.cuda.current_stream(dev)
    l2_bytes = l2_size(dev)

    w = rank_workload(args.config, rank)
    T, H, D = w.q.shape
    R = DeviceWorkload(w, dev, stream, args.partition_size, args.cascade, l2_bytes)
    R.separate_write = args.separate_write
    W = max(3, args.warmup)
    for k in range(W):
        R.step(k=k)
    torch.cuda.synchronize(dev)

    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    # untimed steps for ~0.4 s before the timed region, so that the clock
    # sampler sees the GPU under this load
    soak_steps, t_soak = 0, time.perf_counter()
    while time.perf_counter() - t_soak < 0.4:
        for k in range(50):
            R.step(k=k)
        soak_steps += 50
        torch.cuda.synchronize(dev)

    # ---- device-resident timed region -------------------------------------
    K = args.steps
    if dist is not None:
        dist.barrier()
    total_ms = R.timed(lambda k: R.step(k=k), K)
    step_host_us = R.last_host_us
    # the attention call alone, K calls back to back (the roofline's kernel
    # time: its average launch duration over this region), in three regions:
    # the median region counts, so that one region disturbed on the host
    # cannot set it; all three are reported
    attn_regions_ms = [R.timed(lambda k: R.attend(k=k), K) / K for _ in range(3)]
    attn_host_us = R.last_host_us
    attn_avg_ms = statistics.median(attn_regions_ms)
    if dist is not None:
        dist.barrier()
    # spread of single calls, each between its own pair of events (which
    # serialise it against its neighbours, so these run a little longer)
    NP = min(K, 200)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(NP)]
    for k in range(NP):
        R.attend(ev=evs[k], k=k)
    torch.cuda.synchronize(dev)
    attn_ms = [a.elapsed_time(b) for a, b in evs]

    # ---- end-to-end: inputs from pinned host memory, output back -----------
    # Every step copies all of its inputs from pinned host memory and reads
    # its output back, pipelined the way a serving loop runs: two device
    # buffer sets, the inputs of step k+1 copied (one stream) and the output
    # of step k-1 read back (another) while step k's kernels run; the steps'
    # kernels stay in order on the compute stream (they share the pool). At
    # least 200 steps, so that the pipeline's fill does not set the figure.
    E = args.e2e_steps if args.e2e_steps is not None else max(200, K // 4)
    E = max(E, 1)
    bufs = [(R.d_buf, R.d), R.device_set()]
    results = [(R.out, R.lse), (torch.empty_like(R.out), torch.empty_like(R.lse))]
    out_hosts = [torch.empty((T, H, D), dtype=torch.float32).pin_memory() for _ in range(2)]
    h2d = R.total_in
    d2h = out_hosts[0].numel() * out_hosts[0].element_size()
    copy_in, copy_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    landed = [torch.cuda.Event(), torch.cuda.Event()]   # inputs of the set copied in
    used = [torch.cuda.Event(), torch.cuda.Event()]     # the step's kernels are done with the set
    read = [torch.cuda.Event(), torch.cuda.Event()]     # the set's output is back on the host
    e_start, e_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    e_start.record(stream)
    copy_in.wait_stream(stream)
    copy_out.wait_stream(stream)
    for k in range(E):
        sb = k % 2
        if k >= 2:
            copy_in.wait_event(used[sb])
        with torch.cuda.stream(copy_in):
            bufs[sb][0].copy_(R.host_buf, non_blocking=True)
        landed[sb].record(copy_in)
        stream.wait_event(landed[sb])
        if k >= 2:
            stream.wait_event(read[sb])
        R.step(bufs[sb][1], res=results[sb], k=k)
        used[sb].record(stream)
        copy_out.wait_event(used[sb])
        with torch.cuda.stream(copy_out):
            out_hosts[sb].copy_(results[sb][0], non_blocking=True)
        read[sb].record(copy_out)
    for sb in range(min(E, 2)):
        stream.wait_event(read[sb])
    e_stop.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e_start.elapsed_time(e_stop)

    # ---- the other workloads of the hot path, device-resident --------------
    # (each at least 200 steps and 200 calls after at least 10 warm-up steps:
    # they are cheap, and a few calls right after switching workloads would
    # set their figures)
    KE, WE = max(K, 200), max(W, 10)
    extras = {}
    extra_names = [] if args.extra in ("", "none") else args.extra.split(",")
    for name in extra_names:
        cascade = name.endswith("+cascade")
        base = name[:-len("+cascade")] if cascade else name
        if base == args.config and cascade == args.cascade:
            continue
        del bufs, results
        torch.cuda.empty_cache()
        we = rank_workload(base, rank)
        RE = DeviceWorkload(we, dev, stream, -1, cascade, l2_bytes)
        RE.separate_write = args.separate_write
        for k in range(WE):
            RE.step(k=k)
        if dist is not None:
            dist.barrier()
        e_total = RE.timed(lambda k: RE.step(k=k), KE)
        e_attn = statistics.median(RE.timed(lambda k: RE.attend(k=k), KE) for _ in range(3))
        t = max_over_ranks({"total_ms": e_total, "attn_ms": e_attn}, dist, dev)
        step_ms, attn_e_ms = t["total_ms"] / KE, t["attn_ms"] / KE
        roof, pre = roofline_and_prefill(we, attn_e_ms, RE.ci)
        extras[name] = {
            "num_seqs": we.num_seqs, "num_tokens": we.num_tokens,
            "kv_bytes_per_step": we.kv_bytes(), "step_us": step_ms * 1e3,
            "kv_gbs": job_throughput(world, we.kv_bytes(), step_ms),
            "seqs_per_s": world * we.num_seqs / (step_ms * 1e-3),
            "query_tokens_per_s": world * we.num_tokens / (step_ms * 1e-3),
            "attention_us": attn_e_ms * 1e3, "roofline": roof, "prefill": pre,
            "l2": workload_config(we, -1, world, RE.n_pools, l2_bytes)["l2"],
            "steps": KE, "warmup": WE,
            "gpu_launches": RE.launches_per_step() * KE + (RE.launches_per_step() - 1) * 3 * KE}
        del RE, we
        bufs, results = None, None
        torch.cuda.empty_cache()
    clocks = sampler.stop()

    # ---- reduce over ranks --------------------------------------------------
    slowest = max_over_ranks({"total_ms": total_ms, "e2e_ms": e2e_ms, "attn_avg_ms": attn_avg_ms},
                             dist, dev)
    total_ms, e2e_ms, attn_avg_ms = slowest["total_ms"], slowest["e2e_ms"], slowest["attn_avg_ms"]

    kv_bytes = w.kv_bytes()
    ms_per_step = total_ms / K
    value = job_throughput(world, kv_bytes, ms_per_step)
    e2e_value = job_throughput(world, kv_bytes, e2e_ms / E)
    peak, _ = hbm_peak()
    roof, prefill_line = roofline_and_prefill(w, attn_avg_ms, R.ci)
    roof["traffic"] = profiled_traffic(args.config)
    cpu = None
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        sample, desc = oracle_sample(w)
        sec, cores, n = oracle_step_seconds(sample, args.cpu_seconds)
        sec1, _, n1 = oracle_step_seconds(sample, args.cpu_seconds / 4, threads=1)
        cpu = {"value": sample.kv_bytes() / sec / 1e9, "unit": "GB/s", "cores": cores,
               "kind": "oracle", "sample": f"{desc}; {n} oracle steps, median",
               "seqs_per_s": sample.num_seqs / sec,
               "single_core": {"value": sample.kv_bytes() / sec1 / 1e9, "unit": "GB/s",
                               "steps": n1}}
    if rank == 0:
        # the headline step (K) and attention calls (3 x K), single calls (NP) and
        # e2e steps (E), plus each extra workload's KE steps and 3 x KE calls
        launches = R.launches_per_step()
        line = {
            "metric": "paged decode attention KV GB/s", "value": value, "unit": "GB/s",
            "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": ms_per_step, "host_enqueue_us_per_step": step_host_us,
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "seqs_per_s": world * w.num_seqs / (ms_per_step * 1e-3),
            # one attention layer per step; a 32-layer model's decode step
            # would repeat it 32 times
            "seqs_per_s_32_layers": world * w.num_seqs / (ms_per_step * 1e-3) / 32,
            "attention_us": {"back_to_back_mean": attn_avg_ms * 1e3,
                             "back_to_back_regions": [x * 1e3 for x in attn_regions_ms],
                             "host_enqueue_us_per_call": attn_host_us,
                             "single_call_events": {
                                 "calls": len(attn_ms),
                                 "p10": 1e3 * float(np.percentile(attn_ms, 10)),
                                 "p50": 1e3 * float(np.percentile(attn_ms, 50)),
                                 "p90": 1e3 * float(np.percentile(attn_ms, 90))}},
            "pct_of_hbm_peak": 100.0 * value / world / peak,
            "config": workload_config(w, args.partition_size, world, R.n_pools, l2_bytes),
            "roofline": roof,
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": E, "ms_per_step": e2e_ms / E,
                    "copies": "pinned host, one copy of all inputs in and one of the output "
                              "out per step; step k+1's inputs and step k-1's output move "
                              "while step k runs (two device buffer sets)"},
            "prefill": prefill_line,
            "gpu_launches": (launches * K + (launches - 1) * (3 * K + NP) + launches * E
                             + sum(x["gpu_launches"] for x in extras.values())),
            "workloads": extras,
            "clocks": dict(clocks, soak_steps_before_timing=soak_steps),
            "cpu_baseline": cpu,
        }
        line["config"]["step"] = ("pkv_kv_cache_write + " + ("pkv_cascade_decode" if R.ci is not None
                                                              else "pkv_paged_attention_varlen")
                                  if R.ci is not None or R.separate_write
                                  else "pkv_paged_attention_varlen_append (KV write + attention)")
        if R.ci is not None:
            line["config"]["attention"] = "cascade: each shared prefix read once per group"
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
