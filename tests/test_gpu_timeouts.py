"""Bounded waits that run out (needs a GB300).

Every wait in the kernels is bounded; when one runs out the kernel sets
PKV_DEV_TIMEOUT, lets its copies and products in flight finish, frees its
tensor memory and returns, and the context stays usable. No ordinary input
makes a wait run out, so these tests build a test variant of the library
(PKV_TEST_HOLD_ARRIVAL, a 20 ms wait limit) in which one barrier arrival can
be held back on request: in the decode kernel one warp withholds the copy of
one chunk; in the prefill kernel one softmax warp withholds its P-ready
arrival, so the MMA thread's wait runs out and the CTA unwinds (abort flag,
drain, tensor memory freed, work tickets handed back). Each test then checks
the status bit, that the workspace's work tickets are zero again, and that an
ordinary call right after, through the same library, matches the oracle.
"""
import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import pytest
import torch

from paged_kv_cache_varlen_gb300 import binding as pkv
from paged_kv_cache_varlen_gb300 import build as pkv_build
from paged_kv_cache_varlen_gb300 import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hold_lib(tmp_path_factory):
    out = tmp_path_factory.mktemp("hold_build")
    defines = ["-DPKV_TEST_HOLD_ARRIVAL", "-DPKV_WAIT_TIMEOUT_NS=20000000ull"]

    def comp(src):
        obj = str(out / (os.path.splitext(src)[0] + ".o"))
        cmd = [pkv_build.nvcc(), *pkv_build.NVCC_FLAGS, *defines, "-c",
               os.path.join(pkv_build.CSRC, src), "-o", obj]
        subprocess.run(cmd, check=True, capture_output=True)
        return obj

    with ThreadPoolExecutor(len(pkv_build.SOURCES)) as ex:
        objs = list(ex.map(comp, pkv_build.SOURCES))
    lib_path = str(out / "libpkv_hold.so")
    subprocess.run([pkv_build.nvcc(), *pkv_build.ARCH, "-shared", "-o", lib_path, *objs,
                    "-cudart", "static"], check=True, capture_output=True)
    lib = pkv.load_library(lib_path)
    for name in ("pkv_test_hold_decode", "pkv_test_hold_prefill"):
        getattr(lib, name).restype = ctypes.c_int
        getattr(lib, name).argtypes = [ctypes.c_int]
    saved = pkv._handle
    pkv._handle = lib  # the binding's calls go to the test variant
    try:
        yield lib
    finally:
        pkv._handle = saved


def _run(w, dev, ws):
    out = torch.full(tuple(dev.q.shape), float("nan"), device="cuda")
    lse = torch.full(tuple(dev.q.shape[:2]), float("nan"), device="cuda")
    dev.status.zero_()
    pkv.paged_attention_varlen(dev.q, dev.pool, dev.table, dev.cu, dev.lens, w.max_query_len,
                               w.max_seq_len, out=out, out_lse=lse, scale=w.scale, workspace=ws,
                               dev_status=dev.status)
    return out, lse, dev.dev_status()


@pytest.mark.parametrize("kernel", ["decode", "prefill"])
def test_a_wait_that_runs_out_is_reported_and_the_next_call_is_right(oracle, hold_lib, kernel):
    # decodes (first CTA: request 0, KV head 0, partition 0, at least two
    # chunks per warp) and, for the prefill case, a 300-query chunk
    if kernel == "decode":
        w = wl.build("hold", [2000, 700, 130], [1, 1, 1], 32, 8, 128, seed=81)
    else:
        w = wl.build("hold", [800, 2000, 130], [300, 1, 1], 32, 8, 128, seed=82)
    ref_pool = oracle.kv_cache_write(w.pool, w.k_new, w.v_new, w.slot_mapping)
    dev = gu.DeviceStep(w)
    dev.write()
    assert dev.dev_status() == 0
    need = pkv.attention_workspace_size(w.num_seqs, w.num_tokens, 32, 8, 128, w.max_seq_len, -1)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    setter = hold_lib.pkv_test_hold_decode if kernel == "decode" else hold_lib.pkv_test_hold_prefill
    assert setter(1) == 0
    try:
        _, _, status = _run(w, dev, ws)
    finally:
        assert setter(0) == 0
    assert status & pkv.DEV_TIMEOUT, status
    assert int(ws[-256:].count_nonzero()) == 0, "work tickets not handed back"
    out, lse, status = _run(w, dev, ws)
    assert status == 0
    ref_o, ref_l = oracle.paged_attention(w.q, ref_pool, w.block_table, w.cu_seqlens, w.seq_lens,
                                          w.scale)
    gu.compare(out, lse, ref_o, ref_l)
