"""pa_decode_noalloc: decode attention for callers that cannot allocate.

Some callers may not allocate device memory at all -- an engine that reserved
all GPU memory up front, code that must not block on an allocator, a plugin
whose host owns the device memory.  pa_decode_noalloc serves them with a fixed
scratch array inside the library instead of a caller-provided workspace.  These
tests call it through the C ABI and check that it gives exactly what pa_decode
gives (the same kernels and partition size on the same inputs, so the same
bits), and the oracle's result within the 2e-3 bar, on two calls in a row,
since the array keeps the previous call's contents.  They also check that a
call allocates nothing, and that the first call in a fresh process works.
The file is named to be collected last; it also passes when run alone in a
fresh process.
"""
import ctypes
import os
import subprocess
import sys
import textwrap

import pytest
import torch

from paged_kv_cache_132_gb300 import api, native, workloads
from steps import max_violation, oracle_decode, oracle_pools

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _library():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    native.load()


def _stepped(w):
    """Pools after the step's copies and cache write (every context includes
    its newest token, whose slot holds NaN until then)."""
    k, v = w.k_cache.clone(), w.v_cache.clone()
    if w.copy_pairs.numel():
        api.copy_blocks([k], [v], w.copy_pairs)
    api.reshape_and_cache(w.new_key, w.new_value, k, v, w.slot_mapping)
    return k, v


@pytest.mark.parametrize("name,kwargs,partition", [
    ("tiny", {}, 0),
    ("opt13b", {"num_seqs": 16}, 0),
    ("llama8b", {"num_seqs": 64}, 1024),
    ("long_context", {"num_seqs": 2, "block_size": 16}, 512),
])
def test_noalloc_matches_decode_twice(name, kwargs, partition):
    w = workloads.make(name, device="cuda", **kwargs)
    k, v = _stepped(w)
    max_ctx = int(w.context_lens.max())
    need = api.decode_workspace_size(w.num_seqs, w.num_heads, max_ctx, partition, w.head_dim)
    assert need <= native.NOALLOC_SCRATCH_BYTES, "test batch must fit the static scratch"
    ref = api.decode(w.query, k, v, w.block_tables, w.context_lens, w.scale, max_context_len=max_ctx,
                     partition_size=partition)
    assert api.get_device_error() == (0, 0)
    kref, vref = oracle_pools(w)
    exact = oracle_decode(w, kref, vref)
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        api.decode_noalloc(w.query, k, v, w.block_tables, w.context_lens, w.scale, out=out,
                           max_context_len=max_ctx, partition_size=partition)
        assert api.get_device_error() == (0, 0)
        assert torch.equal(out, ref), "pa_decode_noalloc differs from pa_decode on the same inputs"
        assert max_violation(out, exact) <= 0.0, "pa_decode_noalloc is outside the 2e-3 bar of the oracle"


def test_noalloc_call_allocates_nothing():
    w = workloads.make("llama8b", device="cuda", num_seqs=32)
    k, v = _stepped(w)
    out = torch.empty(w.num_seqs, w.num_heads, w.head_dim, device="cuda")
    run = lambda: api.decode_noalloc(w.query, k, v, w.block_tables, w.context_lens, w.scale, out=out,
                                     max_context_len=w.max_context_len, partition_size=512)
    run()  # the first call on the device does the one-time set-up
    torch.cuda.synchronize()
    before = torch.cuda.mem_get_info()
    for _ in range(3):
        run()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info() == before, "a call changed the device's free memory"
    assert api.get_device_error() == (0, 0)


def test_noalloc_sizes_with_the_partition_that_runs():
    """A batch whose workspace fits the array only at the 512-token partition
    that the automatic choice picks for it (at 256 it would not): accepted,
    and identical to pa_decode."""
    ctx = [4096] + [int(x) for x in torch.randint(16, 4097, (127,), generator=torch.Generator().manual_seed(3))]
    w = workloads.custom(ctx, num_heads=32, num_kv_heads=8, head_dim=128, block_size=16, dtype=torch.bfloat16,
                         device="cuda")
    assert api.decode_workspace_size(128, 32, 4096, 256, 128) > native.NOALLOC_SCRATCH_BYTES
    assert api.decode_workspace_size(128, 32, 4096, 512, 128) <= native.NOALLOC_SCRATCH_BYTES
    k, v = _stepped(w)
    ref = api.decode(w.query, k, v, w.block_tables, w.context_lens, w.scale, max_context_len=4096)
    out = torch.empty_like(ref)
    api.decode_noalloc(w.query, k, v, w.block_tables, w.context_lens, w.scale, out=out, max_context_len=4096)
    assert api.get_device_error() == (0, 0)
    assert torch.equal(out, ref)


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


FRESH = textwrap.dedent("""
    import ctypes, sys
    sys.path.insert(0, {root!r})
    import torch
    from paged_kv_cache_132_gb300 import api, native, workloads
    lib = native.load()
    torch.cuda.init()
    # set-up call: no sequences, nothing launched
    k0 = torch.zeros(1, 2, 16, 64, device="cuda")
    desc = api.cache_desc(k0)
    rc = lib.pa_decode_noalloc(None, 0, None, None, None, ctypes.byref(desc), None, 1, None, 0, 0, 2, 2,
                               0.125, 0, None)
    assert rc == 0, rc
    w = workloads.make("llama8b", device="cuda", num_seqs=16)
    k, v = w.k_cache.clone(), w.v_cache.clone()
    api.reshape_and_cache(w.new_key, w.new_value, k, v, w.slot_mapping)
    out = torch.empty(16, 32, 128, device="cuda")
    # the library's first decode in this process is the allocation-free one
    api.decode_noalloc(w.query, k, v, w.block_tables, w.context_lens, w.scale, out=out,
                       max_context_len=w.max_context_len)
    assert api.get_device_error() == (0, 0)
    ref = api.decode(w.query, k, v, w.block_tables, w.context_lens, w.scale, max_context_len=w.max_context_len)
    assert torch.equal(out, ref)
    print("fresh-process-ok", flush=True)
""")


def test_noalloc_first_call_in_a_fresh_process():
    r = subprocess.run([sys.executable, "-c", FRESH.format(root=ROOT)], cwd=ROOT, timeout=300,
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "fresh-process-ok" in r.stdout
