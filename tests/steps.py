"""One decode step on both sides: the library (through the C ABI) and the oracle.

The step is the one every workload describes: copy-on-write copies, then the
cache write of the new tokens, then decode attention over the updated pools.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
from paged_kv_cache_132_gb300 import api

CODE = {torch.float32: O.F32, torch.float16: O.F16, torch.bfloat16: O.BF16}
ATOL = 2e-3


def bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    return t.view(torch.int32).numpy() if t.dtype == torch.float32 else t.view(torch.int16).numpy()


def gpu_step(w, *, partition_size=None, out_dtype=torch.float32, max_context_len=None):
    """Run the step on the GPU; returns (k_pool, v_pool, out, status, code)."""
    k = w.k_cache.clone()
    v = w.v_cache.clone()
    if w.copy_pairs.numel():
        api.copy_blocks([k], [v], w.copy_pairs)
    api.reshape_and_cache(w.new_key, w.new_value, k, v, w.slot_mapping)
    out = api.decode(w.query, k, v, w.block_tables, w.context_lens, w.scale, out_dtype=out_dtype,
                     max_context_len=w.max_context_len if max_context_len is None else max_context_len,
                     partition_size=w.partition_size if partition_size is None else partition_size)
    status, code = api.get_device_error()
    return k, v, out, status, code


def oracle_pools(w):
    """The oracle's pools after the step's copies and writes (numpy bits)."""
    orc = O.get()
    k = bits(w.k_cache).copy()
    v = bits(w.v_cache).copy()
    if w.copy_pairs.numel():
        orc.copy_blocks([k], [v], w.copy_pairs.cpu().numpy())
    orc.reshape_and_cache(bits(w.new_key), bits(w.new_value), k, v, w.slot_mapping.cpu().numpy())
    return k, v


def oracle_decode(w, k_bits, v_bits, seqs=None, threads=0):
    """fp64 attention for all sequences, or for the listed ones."""
    orc = O.get()
    q = w.query.cpu()
    tables = w.block_tables.cpu().numpy()
    ctx = w.context_lens.cpu().numpy()
    if seqs is not None:
        idx = torch.as_tensor(seqs, dtype=torch.int64)
        q = q[idx]
        tables = tables[np.asarray(seqs)]
        ctx = ctx[np.asarray(seqs)]
    return orc.decode(bits(q), k_bits, v_bits, CODE[w.dtype], tables, ctx, w.num_kv_heads, w.scale,
                      num_threads=threads)


def pools_equal(gpu_pool: torch.Tensor, oracle_bits: np.ndarray) -> bool:
    return np.array_equal(bits(gpu_pool), oracle_bits)


def half_ulp(x: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """Half a unit in the last place of |x| in the output dtype."""
    if dtype == torch.float32:
        return np.zeros_like(x)
    mant = 10 if dtype == torch.float16 else 7
    ax = np.maximum(np.abs(x), 2.0 ** -14 if dtype == torch.float16 else 2.0 ** -126)
    return 0.5 * 2.0 ** (np.floor(np.log2(ax)) - mant)


def max_violation(out: torch.Tensor, ref: np.ndarray) -> float:
    """max(|out - ref| - tolerance); <= 0 means every element is within it."""
    got = out.detach().float().cpu().numpy().astype(np.float64)
    tol = ATOL + half_ulp(ref, out.dtype)
    if not np.all(np.isfinite(got)):
        return float("inf")
    return float(np.max(np.abs(got - ref) - tol)) if got.size else 0.0
