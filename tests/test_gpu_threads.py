"""First calls from two host threads at once (needs a GB300).

The kernels' shared-memory limits are raised once per device, under a lock.
In a fresh process (so that nothing has launched yet), two host threads make
their first prefill-bearing attention calls at the same moment, each on its
own stream with its own workspace; both must succeed and give bitwise the
same outputs as a later call from the main thread.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r'''
import sys, threading
sys.path.insert(0, sys.argv[1])
import torch
from paged_kv_cache_varlen_gb300 import binding as pkv
from paged_kv_cache_varlen_gb300 import workloads as wl
from tests import gpu_util as gu

torch.cuda.init()
w = wl.build("threads", [3000, 700, 1200], [1, 1, 400], 32, 8, 128, seed=61)
dev = gu.DeviceStep(w)
dev.write()
torch.cuda.synchronize()
start = threading.Barrier(2)
results, errors = [None, None], []

def worker(k):
    try:
        torch.cuda.set_device(0)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            out = torch.full(tuple(dev.q.shape), float("nan"), device="cuda")
            lse = torch.full(tuple(dev.q.shape[:2]), float("nan"), device="cuda")
            ws = torch.zeros(pkv.attention_workspace_size(w.num_seqs, w.num_tokens, 32, 8, 128,
                                                          w.max_seq_len, -1),
                             dtype=torch.uint8, device="cuda")
            s.synchronize()
            start.wait()
            pkv.paged_attention_varlen(dev.q, dev.pool, dev.table, dev.cu, dev.lens,
                                       w.max_query_len, w.max_seq_len, out=out, out_lse=lse,
                                       scale=w.scale, workspace=ws, stream=s)
        s.synchronize()
        results[k] = (out, lse)
    except Exception as e:  # reported by the main thread
        errors.append(repr(e))

ts = [threading.Thread(target=worker, args=(k,)) for k in range(2)]
for t in ts:
    t.start()
for t in ts:
    t.join()
assert not errors, errors
ref, ref_lse = dev.attend()
torch.cuda.synchronize()
for out, lse in results:
    assert torch.equal(out, ref) and torch.equal(lse, ref_lse)
assert torch.isfinite(ref).all()
print("threads ok")
'''


def test_first_calls_from_two_threads_at_once():
    res = subprocess.run([sys.executable, "-c", SCRIPT, ROOT], capture_output=True, text=True,
                         timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-4000:]
    assert "threads ok" in res.stdout
