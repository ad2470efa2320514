"""Python binding of the C ABI: argument marshalling only.

Every function takes CUDA tensors, checks their shapes and dtypes, and calls
the same-named entry point of ``libpa.so`` on the current (or given) stream.
All computation happens in the library's kernels; nothing here falls back to
PyTorch or the CPU.  PyTorch provides device memory and streams.
"""
from __future__ import annotations

import contextlib
import ctypes
from typing import Iterator, Optional, Sequence, Tuple

import torch

from . import native
from .native import CacheDesc, PaError

DTYPE_CODE = {torch.float32: native.PA_F32, torch.float16: native.PA_F16, torch.bfloat16: native.PA_BF16}


# The current stream's raw handle without building a Stream object (a few
# microseconds per call saved; decode is called once per layer per step).
_raw_current_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> ctypes.c_void_p:
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream)
    if _raw_current_stream is not None:
        return ctypes.c_void_p(_raw_current_stream(torch.cuda.current_device()))
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _require(cond: bool, msg: str) -> None:
    if not cond:
        raise ValueError(msg)


def _check_cuda(*tensors: torch.Tensor) -> None:
    for t in tensors:
        _require(t.is_cuda, "tensors must be on a CUDA device")
        _require(t.is_contiguous(), "tensors must be contiguous")


def cache_desc(k_cache: torch.Tensor) -> CacheDesc:
    _require(k_cache.dim() == 4, "a pool is [num_blocks][num_kv_heads][block_size][head_dim]")
    _require(k_cache.dtype in DTYPE_CODE, f"unsupported cache dtype {k_cache.dtype}")
    nb, hkv, bs, d = k_cache.shape
    return CacheDesc(nb, hkv, bs, d, DTYPE_CODE[k_cache.dtype])


def _raise(status: int, what: str) -> None:
    if status != native.PA_OK:
        raise PaError(status, what)


def reshape_and_cache(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      slot_mapping: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> None:
    """Write key/value [T][Hkv][d] into the pools at slot_mapping[t] (< 0: skip)."""
    lib = native.load()
    _check_cuda(key, value, k_cache, v_cache, slot_mapping)
    _require(k_cache.shape == v_cache.shape and k_cache.dtype == v_cache.dtype, "K and V pools must match")
    _require(key.dtype == k_cache.dtype and value.dtype == k_cache.dtype, "key/value dtype must match the pools")
    _require(key.dim() == 3 and key.shape == value.shape, "key/value are [num_tokens][num_kv_heads][head_dim]")
    _require(tuple(key.shape[1:]) == (k_cache.shape[1], k_cache.shape[3]), "key/value heads or head_dim mismatch")
    _require(slot_mapping.dtype == torch.int64 and slot_mapping.numel() == key.shape[0], "slot_mapping is int64 [T]")
    desc = cache_desc(k_cache)
    _raise(lib.pa_reshape_and_cache(key.data_ptr(), value.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                    slot_mapping.data_ptr(), key.shape[0], ctypes.byref(desc),
                                    _stream_ptr(stream)), "pa_reshape_and_cache")


class PreparedCacheWrite:
    """A pa_reshape_and_cache call whose arguments are checked and marshalled
    once: for a serving loop that writes each step's new tokens from the same
    buffers (new contents, same tensors) into the same pools.  Each call is
    then one C-ABI call.  The tensors are kept referenced; their shapes,
    dtypes, devices and storage must not change while the object is used."""

    def __init__(self, key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                 slot_mapping: torch.Tensor):
        self._lib = native.load()
        _check_cuda(key, value, k_cache, v_cache, slot_mapping)
        _require(k_cache.shape == v_cache.shape and k_cache.dtype == v_cache.dtype, "K and V pools must match")
        _require(key.dtype == k_cache.dtype and value.dtype == k_cache.dtype, "key/value dtype must match the pools")
        _require(key.dim() == 3 and key.shape == value.shape, "key/value are [num_tokens][num_kv_heads][head_dim]")
        _require(tuple(key.shape[1:]) == (k_cache.shape[1], k_cache.shape[3]), "key/value heads or head_dim mismatch")
        _require(slot_mapping.dtype == torch.int64 and slot_mapping.numel() == key.shape[0],
                 "slot_mapping is int64 [T]")
        self._desc = cache_desc(k_cache)
        self._keep = (key, value, k_cache, v_cache, slot_mapping)
        self._args = (key.data_ptr(), value.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                      slot_mapping.data_ptr(), key.shape[0], ctypes.byref(self._desc))

    def __call__(self, stream: Optional[torch.cuda.Stream] = None) -> None:
        _raise(self._lib.pa_reshape_and_cache(*self._args, _stream_ptr(stream)), "pa_reshape_and_cache")


def decode_workspace_size(num_seqs: int, num_heads: int, max_context_len: int, partition_size: int = 0,
                          head_dim: int = 128) -> int:
    return int(native.load().pa_decode_workspace_size(num_seqs, num_heads, max_context_len, partition_size,
                                                      head_dim))


def decode(query: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
           context_lens: torch.Tensor, scale: float, *, num_kv_heads: Optional[int] = None,
           out: Optional[torch.Tensor] = None, out_dtype: torch.dtype = torch.float32,
           max_context_len: Optional[int] = None, partition_size: int = 0,
           workspace: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Paged decode attention; returns out [S][H][d].

    ``max_context_len`` is a host-side upper bound of context_lens; when None
    the table capacity (max_blocks_per_seq * block_size) is used, which needs
    no device sync but may size a larger workspace."""
    lib = native.load()
    _check_cuda(query, k_cache, v_cache, block_tables, context_lens)
    _require(query.dim() == 3, "query is [num_seqs][num_heads][head_dim]")
    s, h, d = query.shape
    desc = cache_desc(k_cache)
    _require(k_cache.shape == v_cache.shape and v_cache.dtype == k_cache.dtype, "K and V pools must match")
    _require(query.dtype == k_cache.dtype and d == desc.head_dim, "query dtype/head_dim must match the pools")
    _require(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and block_tables.shape[0] == s,
             "block_tables is int32 [num_seqs][max_blocks]")
    _require(context_lens.dtype == torch.int32 and context_lens.numel() == s, "context_lens is int32 [num_seqs]")
    hkv = desc.num_kv_heads if num_kv_heads is None else num_kv_heads
    max_blocks = block_tables.shape[1]
    if max_context_len is None:
        max_context_len = max_blocks * desc.block_size
    if out is None:
        out = torch.empty((s, h, d), dtype=out_dtype, device=query.device)
    _check_cuda(out)
    _require(out.shape == (s, h, d) and out.dtype in DTYPE_CODE, "out is [num_seqs][num_heads][head_dim]")
    if workspace is None:
        need = decode_workspace_size(s, h, max_context_len, partition_size, d)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=query.device)
    _check_cuda(workspace)
    _raise(lib.pa_decode(out.data_ptr(), DTYPE_CODE[out.dtype], query.data_ptr(), k_cache.data_ptr(),
                         v_cache.data_ptr(), ctypes.byref(desc), block_tables.data_ptr(), max_blocks,
                         context_lens.data_ptr(), s, int(max_context_len), h, hkv, float(scale),
                         int(partition_size), workspace.data_ptr(), workspace.numel(), _stream_ptr(stream)),
           "pa_decode")
    return out


class PreparedDecode:
    """A pa_decode call whose arguments are checked and marshalled once: for a
    serving loop that decodes the same buffers every step (new contents, same
    tensors), each call is then one C-ABI call with no per-call argument
    checks.  The tensors are kept referenced; their shapes, dtypes, devices and
    storage must not change while the object is used."""

    def __init__(self, query: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                 block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float, *, out: torch.Tensor,
                 max_context_len: int, workspace: Optional[torch.Tensor] = None,
                 num_kv_heads: Optional[int] = None, partition_size: int = 0):
        self._lib = native.load()
        _check_cuda(query, k_cache, v_cache, block_tables, context_lens, out)
        _require(query.dim() == 3, "query is [num_seqs][num_heads][head_dim]")
        s, h, d = query.shape
        self._desc = cache_desc(k_cache)
        _require(k_cache.shape == v_cache.shape and v_cache.dtype == k_cache.dtype, "K and V pools must match")
        _require(query.dtype == k_cache.dtype and d == self._desc.head_dim, "query dtype/head_dim must match the pools")
        _require(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and block_tables.shape[0] == s,
                 "block_tables is int32 [num_seqs][max_blocks]")
        _require(context_lens.dtype == torch.int32 and context_lens.numel() == s, "context_lens is int32 [num_seqs]")
        _require(out.shape == (s, h, d) and out.dtype in DTYPE_CODE, "out is [num_seqs][num_heads][head_dim]")
        hkv = self._desc.num_kv_heads if num_kv_heads is None else num_kv_heads
        if workspace is None:
            need = decode_workspace_size(s, h, max_context_len, partition_size, d)
            workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=query.device)
        _check_cuda(workspace)
        self._keep = (query, k_cache, v_cache, block_tables, context_lens, out, workspace)
        self.out = out
        self._args = (out.data_ptr(), DTYPE_CODE[out.dtype], query.data_ptr(), k_cache.data_ptr(),
                      v_cache.data_ptr(), ctypes.byref(self._desc), block_tables.data_ptr(), block_tables.shape[1],
                      context_lens.data_ptr(), s, int(max_context_len), h, hkv, ctypes.c_float(float(scale)),
                      int(partition_size), workspace.data_ptr(), workspace.numel())

    def __call__(self, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
        _raise(self._lib.pa_decode(*self._args, _stream_ptr(stream)), "pa_decode")
        return self.out


def prefill(query: torch.Tensor, query_start_loc: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
            block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float, max_query_len: int, *,
            num_kv_heads: Optional[int] = None, out: Optional[torch.Tensor] = None,
            out_dtype: torch.dtype = torch.float32, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Prompt-phase attention of new tokens over a cached prefix; returns
    out [T][H][d].

    Sequence s owns query rows query_start_loc[s] .. query_start_loc[s+1]-1,
    the last n_s of its context_lens[s] cached tokens; row i attends to
    positions 0 .. context_lens[s] - n_s + i.  ``max_query_len`` is a host-side
    upper bound of every n_s."""
    lib = native.load()
    _check_cuda(query, query_start_loc, k_cache, v_cache, block_tables, context_lens)
    _require(query.dim() == 3, "query is [num_tokens][num_heads][head_dim]")
    t, h, d = query.shape
    desc = cache_desc(k_cache)
    _require(k_cache.shape == v_cache.shape and v_cache.dtype == k_cache.dtype, "K and V pools must match")
    _require(query.dtype == k_cache.dtype and d == desc.head_dim, "query dtype/head_dim must match the pools")
    _require(block_tables.dtype == torch.int32 and block_tables.dim() == 2, "block_tables is int32 [S][max_blocks]")
    s = block_tables.shape[0]
    _require(context_lens.dtype == torch.int32 and context_lens.numel() == s, "context_lens is int32 [num_seqs]")
    _require(query_start_loc.dtype == torch.int32 and query_start_loc.numel() == s + 1,
             "query_start_loc is int32 [num_seqs + 1]")
    hkv = desc.num_kv_heads if num_kv_heads is None else num_kv_heads
    if out is None:
        out = torch.empty((t, h, d), dtype=out_dtype, device=query.device)
    _check_cuda(out)
    _require(out.shape == (t, h, d) and out.dtype in DTYPE_CODE, "out is [num_tokens][num_heads][head_dim]")
    _raise(lib.pa_prefill(out.data_ptr(), DTYPE_CODE[out.dtype], query.data_ptr(), query_start_loc.data_ptr(), t,
                          int(max_query_len), k_cache.data_ptr(), v_cache.data_ptr(), ctypes.byref(desc),
                          block_tables.data_ptr(), block_tables.shape[1], context_lens.data_ptr(), s, h, hkv,
                          float(scale), _stream_ptr(stream)), "pa_prefill")
    return out


def copy_blocks(k_caches: Sequence[torch.Tensor], v_caches: Sequence[torch.Tensor], src_dst_pairs: torch.Tensor,
                stream: Optional[torch.cuda.Stream] = None) -> None:
    """Copy-on-write: copy K and V block pairs[i][0] -> pairs[i][1] in every layer."""
    lib = native.load()
    _require(len(k_caches) == len(v_caches) and len(k_caches) > 0, "one K and one V pool per layer")
    _check_cuda(*k_caches, *v_caches, src_dst_pairs)
    _require(src_dst_pairs.dtype == torch.int64 and src_dst_pairs.dim() == 2 and src_dst_pairs.shape[1] == 2,
             "src_dst_pairs is int64 [n][2]")
    desc = cache_desc(k_caches[0])
    for p in list(k_caches) + list(v_caches):
        _require(p.shape == k_caches[0].shape and p.dtype == k_caches[0].dtype, "all pools must match")
    n = len(k_caches)
    kp = (ctypes.c_void_p * n)(*[p.data_ptr() for p in k_caches])
    vp = (ctypes.c_void_p * n)(*[p.data_ptr() for p in v_caches])
    _raise(lib.pa_copy_blocks(kp, vp, n, src_dst_pairs.data_ptr(), src_dst_pairs.shape[0], ctypes.byref(desc),
                              _stream_ptr(stream)), "pa_copy_blocks")


def swap_blocks(src_k: Sequence[torch.Tensor], src_v: Sequence[torch.Tensor], dst_k: Sequence[torch.Tensor],
                dst_v: Sequence[torch.Tensor], src_dst_pairs: torch.Tensor,
                stream: Optional[torch.cuda.Stream] = None) -> None:
    """Copy blocks pairs[i][0] of the source pools to blocks pairs[i][1] of
    the destination pools, every layer, one launch: GPU <-> page-locked host
    (swap-out / swap-in).  Host pools must be pinned (``pin_memory()``)."""
    lib = native.load()
    n = len(src_k)
    _require(n > 0 and len(src_v) == n and len(dst_k) == n and len(dst_v) == n, "one pool per layer on each side")
    pools = list(src_k) + list(src_v) + list(dst_k) + list(dst_v)
    for p in pools:
        _require(p.is_contiguous(), "pools must be contiguous")
        _require(p.is_cuda or p.is_pinned(), "host pools must be in page-locked (pinned) memory")
        _require(p.dtype == src_k[0].dtype and tuple(p.shape[1:]) == tuple(src_k[0].shape[1:]),
                 "pools must share dtype and block shape")
    _require(src_dst_pairs.dtype == torch.int64 and src_dst_pairs.dim() == 2 and src_dst_pairs.shape[1] == 2,
             "src_dst_pairs is int64 [n][2]")
    _require(src_dst_pairs.is_cuda or src_dst_pairs.is_pinned(), "pairs must be on the GPU or pinned")
    _require(src_dst_pairs.is_contiguous(), "pairs must be contiguous")
    desc = cache_desc(src_k[0])
    arr = lambda ts: (ctypes.c_void_p * n)(*[t.data_ptr() for t in ts])
    _raise(lib.pa_swap_blocks(arr(src_k), arr(src_v), src_k[0].shape[0], arr(dst_k), arr(dst_v), dst_k[0].shape[0],
                              n, src_dst_pairs.data_ptr(), src_dst_pairs.shape[0], ctypes.byref(desc),
                              _stream_ptr(stream)), "pa_swap_blocks")


def get_device_error(stream: Optional[torch.cuda.Stream] = None) -> Tuple[int, int]:
    """(status, PA_DEVERR_* mask); synchronises the stream and clears the word."""
    code = ctypes.c_int32(0)
    status = native.load().pa_get_device_error(_stream_ptr(stream), ctypes.byref(code))
    return int(status), int(code.value)


def decode_noalloc(query: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                   context_lens: torch.Tensor, scale: float, *, out: torch.Tensor, max_context_len: int,
                   num_kv_heads: Optional[int] = None, partition_size: int = 0,
                   stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Decode attention through pa_decode_noalloc: for callers that must not
    allocate device memory.  ``out`` must be given (nothing is allocated
    here either); the workspace is the library's fixed array, so the batch must
    fit in it (PA_ERR_WORKSPACE otherwise) and calls that overlap on the GPU
    must be serialised by the caller."""
    lib = native.load()
    _check_cuda(query, k_cache, v_cache, block_tables, context_lens, out)
    s, h, d = query.shape
    desc = cache_desc(k_cache)
    _require(query.dtype == k_cache.dtype and d == desc.head_dim, "query dtype/head_dim must match the pools")
    _require(out.shape == (s, h, d) and out.dtype in DTYPE_CODE, "out is [num_seqs][num_heads][head_dim]")
    hkv = desc.num_kv_heads if num_kv_heads is None else num_kv_heads
    _raise(lib.pa_decode_noalloc(out.data_ptr(), DTYPE_CODE[out.dtype], query.data_ptr(), k_cache.data_ptr(),
                                 v_cache.data_ptr(), ctypes.byref(desc), block_tables.data_ptr(),
                                 block_tables.shape[1], context_lens.data_ptr(), s, int(max_context_len), h, hkv,
                                 float(scale), int(partition_size), _stream_ptr(stream)), "pa_decode_noalloc")
    return out


OPTIONS = {"debug_checks": native.OPT_DEBUG_CHECKS, "decode_kernel_simt": native.OPT_DECODE_KERNEL,
           "drop_first_fill": native.OPT_DROP_FIRST_FILL}


def set_option(name: str, value: bool) -> bool:
    """Set a process-wide library option (pa_set_option); returns the previous
    value.  ``debug_checks``: checked mode (precondition pre-passes that report
    violations through the error word); ``decode_kernel_simt``: CUDA-core
    decode for 16-bit pools; ``drop_first_fill``: test hook of the bounded
    waits."""
    prev = native.load().pa_set_option(OPTIONS[name], 1 if value else 0)
    if prev < 0:
        raise PaError(prev, "pa_set_option")
    return bool(prev)


def get_option(name: str) -> bool:
    value = native.load().pa_get_option(OPTIONS[name])
    if value < 0:
        raise PaError(value, "pa_get_option")
    return bool(value)


@contextlib.contextmanager
def option(name: str, value: bool = True) -> Iterator[None]:
    """``with api.option("debug_checks"):`` -- the option set for the block,
    restored afterwards."""
    prev = set_option(name, value)
    try:
        yield
    finally:
        set_option(name, prev)
