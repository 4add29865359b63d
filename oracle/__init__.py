"""fp64 CPU oracle for paged KV-cache attention (test infrastructure).

This package is TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import it. The GPU library does
not depend on it, and it does not depend on the GPU library.

The arithmetic lives in ``oracle.c`` (plain C, fp64, no tiling); this module
only compiles it with gcc, loads it with ctypes and marshals numpy arrays.
bf16 tensors are passed as their uint16 bit patterns.

Sources are the three pages cited at the top of ``oracle.c``:
page 1 (zizhi168.cn, §02 Paged Attention, §04 Attention, §07),
page 2 (su666666.com, PagedAttention deep-dive, step 4),
page 3 (adg.csdn.net, §1.5 KV-cache sizing).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle.c")
LIBRARY = os.path.join(_HERE, "liboracle.so")

_lock = threading.Lock()
_cache: dict[str, "Oracle"] = {}

CFLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared"]


def compile_oracle(source: str = SOURCE, output: str = LIBRARY) -> str:
    """Compile ``source`` into the shared library ``output`` with gcc."""
    cmd = ["gcc", *CFLAGS, source, "-o", output + ".tmp", "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(output + ".tmp", output)
    return output


def _stale(lib: str, src: str) -> bool:
    return not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(src)


_i32p = ctypes.POINTER(ctypes.c_int32)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_f64p = ctypes.POINTER(ctypes.c_double)


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctype)


class OracleError(RuntimeError):
    pass


_ERRORS = {1: "bad shape", 2: "slot out of range", 3: "block id out of range",
           4: "inconsistent lengths", 5: "out of memory"}


def _check(rc: int):
    if rc != 0:
        raise OracleError(f"oracle rejected its input: {_ERRORS.get(rc, rc)}")


class Oracle:
    """ctypes view of one compiled copy of ``oracle.c``."""

    def __init__(self, path: str):
        self.path = path
        lib = ctypes.CDLL(path)
        self._lib = lib
        lib.oracle_kv_cache_write.restype = ctypes.c_int
        lib.oracle_kv_cache_write.argtypes = [_u16p, _u16p, _u16p, _i32p] + [ctypes.c_int32] * 5
        lib.oracle_paged_attention_rows.restype = ctypes.c_int
        lib.oracle_paged_attention_rows.argtypes = (
            [_f64p, _f64p, _i32p, ctypes.c_int32, _u16p, _u16p, _i32p, ctypes.c_int32,
             _i32p, _i32p] + [ctypes.c_int32] * 7 + [ctypes.c_double, ctypes.c_int64,
                                                      ctypes.c_int64])
        lib.oracle_attention_probs.restype = ctypes.c_int64
        lib.oracle_attention_probs.argtypes = (
            [_f64p, ctypes.c_int32, ctypes.c_int32, _u16p, _u16p, _i32p, ctypes.c_int32,
             _i32p, _i32p] + [ctypes.c_int32] * 7 + [ctypes.c_double])
        lib.oracle_lse_merge.restype = None
        lib.oracle_lse_merge.argtypes = [_f64p, _f64p, _f64p, _f64p, ctypes.c_int32,
                                         ctypes.c_int64, ctypes.c_int32]
        lib.oracle_kv_bytes_per_token.restype = ctypes.c_int64
        lib.oracle_kv_bytes_per_token.argtypes = [ctypes.c_int64] * 4
        lib.oracle_kv_cache_bytes.restype = ctypes.c_int64
        lib.oracle_kv_cache_bytes.argtypes = [ctypes.c_int64] * 6
        lib.oracle_set_num_threads.restype = None
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        lib.oracle_get_num_threads.restype = ctypes.c_int
        lib.oracle_get_num_threads.argtypes = []

    # -- threads -----------------------------------------------------------
    def set_num_threads(self, n: int) -> None:
        self._lib.oracle_set_num_threads(int(n))

    def num_threads(self) -> int:
        return int(self._lib.oracle_get_num_threads())

    # -- KV write ----------------------------------------------------------
    def kv_cache_write(self, pool: np.ndarray, k_new: np.ndarray, v_new: np.ndarray,
                       slot_mapping: np.ndarray) -> np.ndarray:
        """Return a copy of ``pool`` [2,NB,BS,Hkv,D] (uint16) after the write."""
        assert pool.dtype == np.uint16 and pool.ndim == 5 and pool.shape[0] == 2
        _, nb, bs, hkv, d = pool.shape
        out = np.ascontiguousarray(pool).copy()
        k = np.ascontiguousarray(k_new, dtype=np.uint16)
        v = np.ascontiguousarray(v_new, dtype=np.uint16)
        slots = np.ascontiguousarray(slot_mapping, dtype=np.int32)
        t = slots.shape[0]
        assert k.shape == (t, hkv, d) and v.shape == (t, hkv, d)
        _check(self._lib.oracle_kv_cache_write(_ptr(out, _u16p), _ptr(k, _u16p), _ptr(v, _u16p),
                                               _ptr(slots, _i32p), t, nb, bs, hkv, d))
        return out

    # -- attention ---------------------------------------------------------
    def paged_attention(self, q, pool, block_table, cu_seqlens, seq_lens, scale,
                        rows=None, key_begin: int = 0, key_end: int = -1):
        """Attention rows for flattened tokens ``rows`` (default: all tokens).

        Returns ``(out, lse)``: out [R,H,D] float64, lse [R,H] float64.
        """
        q = np.ascontiguousarray(q, dtype=np.uint16)
        pool = np.ascontiguousarray(pool, dtype=np.uint16)
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        t, h, d = q.shape
        _, nb, bs, hkv, d2 = pool.shape
        assert d == d2
        b = sl.shape[0]
        if bt.ndim == 1:
            bt = bt.reshape(b, -1)
        max_blocks = bt.shape[1] if bt.ndim == 2 else 0
        rows = np.arange(t, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
        out = np.zeros((rows.shape[0], h, d), dtype=np.float64)
        lse = np.zeros((rows.shape[0], h), dtype=np.float64)
        if bt.size == 0:
            bt = np.zeros((max(b, 1), 1), dtype=np.int32)
        _check(self._lib.oracle_paged_attention_rows(
            _ptr(out, _f64p), _ptr(lse, _f64p), _ptr(rows, _i32p), rows.shape[0],
            _ptr(q, _u16p), _ptr(pool, _u16p), _ptr(bt, _i32p), max_blocks,
            _ptr(cu, _i32p), _ptr(sl, _i32p), b, t, h, hkv, d, bs, nb, float(scale),
            int(key_begin), int(key_end)))
        return out, lse

    def attention_probs(self, q, pool, block_table, cu_seqlens, seq_lens, scale, t: int, h: int):
        """Softmax row P (float64, one entry per visible key) of token t, head h."""
        q = np.ascontiguousarray(q, dtype=np.uint16)
        pool = np.ascontiguousarray(pool, dtype=np.uint16)
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        nt, nh, d = q.shape
        _, nb, bs, hkv, _ = pool.shape
        b = sl.shape[0]
        probs = np.zeros(int(sl.max()) if b else 1, dtype=np.float64)
        n = self._lib.oracle_attention_probs(
            _ptr(probs, _f64p), int(t), int(h), _ptr(q, _u16p), _ptr(pool, _u16p),
            _ptr(bt, _i32p), bt.shape[1], _ptr(cu, _i32p), _ptr(sl, _i32p), b, nt, nh, hkv, d,
            bs, nb, float(scale))
        if n < 0:
            _check(-n)
        return probs[:n]

    # -- merge -------------------------------------------------------------
    def lse_merge(self, part_out: np.ndarray, part_lse: np.ndarray):
        """Merge partials part_out [P,R...,D], part_lse [P,R...] -> (out, lse)."""
        po = np.ascontiguousarray(part_out, dtype=np.float64)
        pl = np.ascontiguousarray(part_lse, dtype=np.float64)
        p = po.shape[0]
        d = po.shape[-1]
        row_shape = pl.shape[1:]
        rows = int(np.prod(row_shape)) if row_shape else 1
        assert po.shape[1:-1] == row_shape
        out = np.zeros(row_shape + (d,), dtype=np.float64)
        lse = np.zeros(row_shape, dtype=np.float64)
        self._lib.oracle_lse_merge(_ptr(out, _f64p), _ptr(lse, _f64p), _ptr(po, _f64p),
                                   _ptr(pl, _f64p), p, rows, d)
        return out, lse

    # -- sizing ------------------------------------------------------------
    def kv_bytes_per_token(self, num_layers, num_kv_heads, head_dim, bytes_per_element):
        return int(self._lib.oracle_kv_bytes_per_token(num_layers, num_kv_heads, head_dim,
                                                        bytes_per_element))

    def kv_cache_bytes(self, batch, seq_len, num_layers, num_kv_heads, head_dim,
                       bytes_per_element):
        return int(self._lib.oracle_kv_cache_bytes(batch, seq_len, num_layers, num_kv_heads,
                                                   head_dim, bytes_per_element))


def load(path: str | None = None) -> Oracle:
    """Load the oracle (compiling ``oracle.c`` first if the library is stale)."""
    with _lock:
        if path is None:
            if _stale(LIBRARY, SOURCE):
                compile_oracle()
            path = LIBRARY
        if path not in _cache:
            _cache[path] = Oracle(path)
        return _cache[path]
