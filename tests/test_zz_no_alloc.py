"""pa_decode_noalloc: decode attention for callers that cannot allocate.

Some callers may not allocate device memory at all -- an engine that reserved
all GPU memory up front, code that must not block on an allocator, a plugin
whose host owns the device memory.  pa_decode_noalloc serves them with a fixed
scratch array inside the library instead of a caller-provided workspace.  These
tests call it through the C ABI and check that it gives what pa_decode gives
(within the 2e-3 bar of the parity tests), on two calls in a row, since the
array keeps the previous call's contents.  The file is named to be collected
last; it also passes when run alone in a fresh process.
"""
import ctypes

import pytest
import torch

from paged_kv_cache_132_gb300 import api, native, workloads

pytestmark = pytest.mark.gpu

ATOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _library():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    native.load()


@pytest.mark.parametrize("name,kwargs,partition", [
    ("tiny", {}, 0),
    ("opt13b", {"num_seqs": 16}, 0),
    ("llama8b", {"num_seqs": 64}, 1024),
    ("long_context", {"num_seqs": 2, "block_size": 16}, 512),
])
def test_noalloc_matches_decode_twice(name, kwargs, partition):
    w = workloads.make(name, device="cuda", **kwargs)
    # The step's new tokens go into the cache first (their slots hold NaN
    # until then, and every context includes its newest token).
    k, v = w.k_cache.clone(), w.v_cache.clone()
    if w.copy_pairs.numel():
        api.copy_blocks([k], [v], w.copy_pairs)
    api.reshape_and_cache(w.new_key, w.new_value, k, v, w.slot_mapping)
    max_ctx = int(w.context_lens.max())
    need = api.decode_workspace_size(w.num_seqs, w.num_heads, max_ctx, partition, w.head_dim)
    assert need <= native.NOALLOC_SCRATCH_BYTES, "test batch must fit the static scratch"
    ref = api.decode(w.query, k, v, w.block_tables, w.context_lens, w.scale, max_context_len=max_ctx,
                     partition_size=partition)
    assert torch.isfinite(ref).all()
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        api.decode_noalloc(w.query, k, v, w.block_tables, w.context_lens, w.scale, out=out,
                           max_context_len=max_ctx, partition_size=partition)
        assert api.get_device_error() == (0, 0)
        assert torch.isfinite(out).all()
        assert torch.max(torch.abs(out - ref)).item() <= ATOL


def test_noalloc_rejects_batch_larger_than_scratch():
    # A consistent batch (every tensor sized for it, all ids valid) whose
    # workspace needs more than the array: 4096 sequences with a declared
    # maximum context of 1M tokens.  The call must refuse before launching.
    s, h, d, big = 4096, 4, 64, 1 << 20
    assert api.decode_workspace_size(s, h, big, 0, d) > native.NOALLOC_SCRATCH_BYTES
    k = torch.zeros(1, h, 16, d, device="cuda")
    v = torch.zeros_like(k)
    q = torch.zeros(s, h, d, device="cuda")
    tables = torch.zeros(s, 1, dtype=torch.int32, device="cuda")
    ctx = torch.ones(s, dtype=torch.int32, device="cuda")
    out = torch.zeros(s, h, d, device="cuda")
    desc = api.cache_desc(k)
    status = native.load().pa_decode_noalloc(out.data_ptr(), 0, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                             ctypes.byref(desc), tables.data_ptr(), 1, ctx.data_ptr(), s, big, h,
                                             h, 0.125, 0, None)
    assert status == -3  # PA_ERR_WORKSPACE
    assert torch.count_nonzero(out) == 0  # nothing ran
