"""CPU fp64 oracle for paged decode attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls it, and shares no code with
it.  The arithmetic lives in ``pa_oracle.c`` (plain C, fp64); this module only
compiles it with gcc and marshals numpy arrays into it.

Array conventions (numpy, C-contiguous):
  * 32-bit float data: ``np.float32``; 16-bit data (binary16 or bfloat16):
    the raw bits as ``np.uint16``/``np.int16``, with ``dtype`` telling which.
  * Pools ``[num_blocks][num_kv_heads][block_size][head_dim]``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F32, F16, BF16 = 0, 1, 2

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "pa_oracle.c")
HEADER = os.path.join(_HERE, "pa_oracle.h")
LIB_DIR = os.path.join(_HERE, "lib")
LIB_PATH = os.path.join(LIB_DIR, "libpa_oracle.so")

_lock = threading.Lock()
_default = None


def compile_oracle(source: str = SOURCE, out: str = LIB_PATH, include_dir: str = _HERE) -> str:
    """Compile ``source`` (plain C11, -O2, no fast-math, OpenMP) into ``out``."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared", "-I", include_dir,
           source, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, out)
    return out


def _stale(out: str) -> bool:
    if not os.path.exists(out):
        return True
    built = os.path.getmtime(out)
    return any(os.path.getmtime(p) > built for p in (SOURCE, HEADER))


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        self.path = path
        lib = ctypes.CDLL(path)
        vp, i64, i32, dbl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.orc_elem_to_double.argtypes = [vp, i64, i32]
        lib.orc_elem_to_double.restype = dbl
        lib.orc_reshape_and_cache.argtypes = [vp, vp, vp, vp, vp, i64, i64, i32, i32, i32, i32]
        lib.orc_copy_blocks.argtypes = [vp, vp, i32, vp, i64, i64, i64]
        lib.orc_swap_blocks.argtypes = [vp, vp, i64, vp, vp, i64, i32, vp, i64, i64]
        lib.orc_decode.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, vp, i32, i32, i32, i32,
                                   i32, i64, dbl, i32]
        lib.orc_decode_partitioned.argtypes = [vp, vp, vp, vp, i32, vp, i32, vp, i32, i32, i32,
                                               i32, i32, i64, dbl, i32]
        lib.orc_prefill.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, vp, i32, i32, i32, i32, i32, i64, dbl,
                                    i32]
        lib.orc_max_threads.argtypes = []
        for name in ("orc_reshape_and_cache", "orc_copy_blocks", "orc_swap_blocks", "orc_decode",
                     "orc_decode_partitioned", "orc_prefill", "orc_max_threads"):
            getattr(lib, name).restype = ctypes.c_int
        self.lib = lib

    # -- helpers -----------------------------------------------------------
    @staticmethod
    def _ptr(a: np.ndarray) -> int:
        assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
        return a.ctypes.data

    @staticmethod
    def _check(rc: int, what: str) -> None:
        if rc != 0:
            raise ValueError(f"oracle {what} failed with status {rc}")

    def max_threads(self) -> int:
        return int(self.lib.orc_max_threads())

    def elem_to_double(self, arr: np.ndarray, index: int, dtype: int) -> float:
        return float(self.lib.orc_elem_to_double(self._ptr(arr), index, dtype))

    def elems_to_double(self, arr: np.ndarray, dtype: int) -> np.ndarray:
        flat = np.ascontiguousarray(arr).reshape(-1)
        return np.array([self.elem_to_double(flat, i, dtype) for i in range(flat.size)])

    # -- the three operations ---------------------------------------------
    def reshape_and_cache(self, key, value, k_pool, v_pool, slot_mapping):
        """In place on k_pool/v_pool: the cache write of key/value [T][Hkv][d]."""
        nb, hkv, bs, d = k_pool.shape
        assert key.shape[1:] == (hkv, d) and value.shape == key.shape
        assert key.dtype == k_pool.dtype == value.dtype == v_pool.dtype
        slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        rc = self.lib.orc_reshape_and_cache(self._ptr(key), self._ptr(value), self._ptr(k_pool),
                                            self._ptr(v_pool), self._ptr(slots), slots.size, nb,
                                            hkv, bs, d, key.itemsize)
        self._check(rc, "reshape_and_cache")

    def copy_blocks(self, k_pools, v_pools, pairs):
        """In place on every pool: the copy-on-write copies listed in pairs [n][2]."""
        pairs = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
        nb = k_pools[0].shape[0]
        block_bytes = k_pools[0][0].nbytes
        kp = (ctypes.c_void_p * len(k_pools))(*[self._ptr(p) for p in k_pools])
        vp = (ctypes.c_void_p * len(v_pools))(*[self._ptr(p) for p in v_pools])
        rc = self.lib.orc_copy_blocks(kp, vp, len(k_pools), self._ptr(pairs), pairs.shape[0], nb,
                                      block_bytes)
        self._check(rc, "copy_blocks")

    def swap_blocks(self, src_k, src_v, dst_k, dst_v, pairs):
        """In place on the destination pools: blocks pairs[i][0] of the
        source pools to blocks pairs[i][1] of the destination pools."""
        pairs = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
        n = len(src_k)
        arr = lambda pools: (ctypes.c_void_p * n)(*[self._ptr(q) for q in pools])
        rc = self.lib.orc_swap_blocks(arr(src_k), arr(src_v), src_k[0].shape[0], arr(dst_k), arr(dst_v),
                                      dst_k[0].shape[0], n, self._ptr(pairs), pairs.shape[0],
                                      src_k[0][0].nbytes)
        self._check(rc, "swap_blocks")

    def decode(self, query, k_pool, v_pool, dtype, block_tables, context_lens, num_kv_heads,
               scale, num_threads=1, want_weight_sum=False):
        """fp64 attention output [S][H][d] (and the per-row weight sums)."""
        s, h, d = query.shape
        nb, hkv, bs, d2 = k_pool.shape
        assert d2 == d and hkv == num_kv_heads
        tables = np.ascontiguousarray(block_tables, dtype=np.int32)
        ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
        out = np.zeros((s, h, d), dtype=np.float64)
        wsum = np.zeros((s, h), dtype=np.float64) if want_weight_sum else None
        rc = self.lib.orc_decode(self._ptr(out), self._ptr(wsum) if wsum is not None else None,
                                 self._ptr(query), self._ptr(k_pool), self._ptr(v_pool), dtype,
                                 self._ptr(tables), tables.shape[1] if tables.ndim == 2 else 0,
                                 self._ptr(ctx), s, h, hkv, bs, d, nb, float(scale),
                                 int(num_threads))
        self._check(rc, "decode")
        return (out, wsum) if want_weight_sum else out

    def prefill(self, query, query_start, k_pool, v_pool, dtype, block_tables, context_lens, num_kv_heads, scale,
                num_threads=1):
        """fp64 prefill output [rows][H][d] for query rows [rows][H][d]."""
        rows, h, d = query.shape
        nb, hkv, bs, d2 = k_pool.shape
        assert d2 == d and hkv == num_kv_heads
        qs = np.ascontiguousarray(query_start, dtype=np.int32)
        tables = np.ascontiguousarray(block_tables, dtype=np.int32)
        ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
        assert qs.size == ctx.size + 1 and qs[-1] == rows
        out = np.zeros((rows, h, d), dtype=np.float64)
        rc = self.lib.orc_prefill(self._ptr(out), self._ptr(query), self._ptr(qs), self._ptr(k_pool),
                                  self._ptr(v_pool), dtype, self._ptr(tables), tables.shape[1], self._ptr(ctx),
                                  ctx.size, h, hkv, bs, d, nb, float(scale), int(num_threads))
        self._check(rc, "prefill")
        return out

    def decode_partitioned(self, query, k_pool, v_pool, dtype, block_tables, context_lens,
                           num_kv_heads, scale, partition_size):
        s, h, d = query.shape
        nb, hkv, bs, _ = k_pool.shape
        tables = np.ascontiguousarray(block_tables, dtype=np.int32)
        ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
        out = np.zeros((s, h, d), dtype=np.float64)
        rc = self.lib.orc_decode_partitioned(self._ptr(out), self._ptr(query), self._ptr(k_pool),
                                             self._ptr(v_pool), dtype, self._ptr(tables),
                                             tables.shape[1], self._ptr(ctx), s, h, hkv, bs, d,
                                             nb, float(scale), int(partition_size))
        self._check(rc, "decode_partitioned")
        return out


def get() -> Oracle:
    """The oracle built from this directory's source (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            if _stale(LIB_PATH):
                compile_oracle()
            _default = Oracle(LIB_PATH)
        return _default


def build() -> str:
    """Compile the oracle library in place (used by the build entry point)."""
    return compile_oracle()
