"""Helpers for the GPU parity tests: move a seeded workload to the device,
run one step through the C ABI, and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

from paged_kv_cache_varlen_gb300 import binding as pkv
from paged_kv_cache_varlen_gb300 import workloads as wl

# The attention tolerance: max-abs error 2e-3 against the fp64 oracle
# (bf16 inputs, fp32 accumulation, fp32 output).
ATOL = 2e-3


def bf16_tensor(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


def i32_tensor(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def to_numpy_bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


class DeviceStep:
    """A workload resident on the GPU."""

    def __init__(self, w: wl.Workload, device="cuda"):
        self.w = w
        self.pool = bf16_tensor(w.pool, device)
        self.q = bf16_tensor(w.q, device)
        self.k_new = bf16_tensor(w.k_new, device)
        self.v_new = bf16_tensor(w.v_new, device)
        self.slots = i32_tensor(w.slot_mapping, device)
        self.table = i32_tensor(w.block_table, device)
        self.cu = i32_tensor(w.cu_seqlens, device)
        self.lens = i32_tensor(w.seq_lens, device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def write(self):
        pkv.kv_cache_write(self.pool, self.k_new, self.v_new, self.slots, dev_status=self.status)

    def attend(self, partition_size=-1, q=None, table=None, cu=None, lens=None, pool=None):
        w = self.w
        q = self.q if q is None else q
        out = torch.full(tuple(q.shape), float("nan"), dtype=torch.float32, device=q.device)
        lse = torch.full(tuple(q.shape[:2]), float("nan"), dtype=torch.float32, device=q.device)
        pkv.paged_attention_varlen(
            q, self.pool if pool is None else pool, self.table if table is None else table,
            self.cu if cu is None else cu, self.lens if lens is None else lens,
            w.max_query_len, w.max_seq_len, out=out, out_lse=lse, scale=w.scale,
            partition_size=partition_size, dev_status=self.status)
        return out, lse

    def dev_status(self) -> int:
        torch.cuda.synchronize()
        return int(self.status.item())


def guarded(shape, dtype, guard: int = 8192, device="cuda"):
    """A tensor of `shape` inside a larger buffer whose `guard` elements on
    each side hold a sentinel bit pattern (stands in for a memory checker:
    a kernel that writes outside the tensor changes a sentinel). Returns
    (buffer, view); the view starts guard * itemsize bytes in (a multiple of
    256 for every dtype here)."""
    n = 1
    for d in shape:
        n *= d
    bits = {torch.float32: (torch.int32, 0x7FBADBAD), torch.bfloat16: (torch.int16, 0x7DAD),
            torch.int32: (torch.int32, 0x5EA1ED), torch.uint8: (torch.uint8, 0xA5)}[dtype]
    buf = torch.full((guard + n + guard,), bits[1], dtype=bits[0], device=device)
    view = buf.view(dtype)[guard:guard + n].view(shape)
    return buf, view


def guards_intact(buf: torch.Tensor, n: int, guard: int = 8192) -> bool:
    """True when both sentinel bands of a `guarded` buffer are unchanged."""
    sentinel = buf[0].item()
    return bool(torch.all(buf[:guard] == sentinel) and torch.all(buf[guard + n:] == sentinel))


def compare(out: torch.Tensor, lse: torch.Tensor, ref_out: np.ndarray, ref_lse: np.ndarray,
            rows: np.ndarray | None = None, atol: float = ATOL):
    """Max-abs errors of out and lse (GPU fp32 vs oracle fp64) on `rows`."""
    o = out.cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64)
    if rows is not None:
        o, l = o[rows], l[rows]
    assert np.all(np.isfinite(o)), "non-finite attention output"
    assert np.all(np.isfinite(l)), "non-finite lse"
    err_o = float(np.max(np.abs(o - ref_out))) if o.size else 0.0
    err_l = float(np.max(np.abs(l - ref_lse))) if l.size else 0.0
    assert err_o <= atol, f"max |out - oracle| = {err_o:.3e} > {atol}"
    assert err_l <= atol, f"max |lse - oracle| = {err_l:.3e} > {atol}"
    return err_o, err_l
