"""GPU parity: the library (through the C ABI) against the fp64 oracle.

Cache writes and block copies must match bit for bit over the whole pool;
attention outputs must be within 2e-3 absolute (fp32 output), or 2e-3 plus
half an ulp of the output type.  Workloads fill every stale slot with NaN.
"""
import dataclasses

import numpy as np
import pytest
import torch

from paged_kv_cache_132_gb300 import api, native, workloads
from steps import (ATOL, bits, gpu_step, max_violation, oracle_decode, oracle_pools, pools_equal)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    native.load()  # raises if the library was not built: no fallback


@pytest.fixture(params=["mma", "simt"])
def kernel(request):
    """Run the test with the tensor-core decode kernel (the default for 16-bit
    pools) and again with the CUDA-core one."""
    with api.option("decode_kernel_simt", request.param == "simt"):
        yield request.param


def _check_step(w, **kw):
    k, v, out, status, code = gpu_step(w, **kw)
    assert status == 0 and code == 0, f"device error {status} / {code:#x}"
    kref, vref = oracle_pools(w)
    assert pools_equal(k, kref), "K pool differs from the oracle"
    assert pools_equal(v, vref), "V pool differs from the oracle"
    ref = oracle_decode(w, kref, vref)
    err = np.max(np.abs(out.float().cpu().numpy() - ref))
    assert max_violation(out, ref) <= 0.0, f"max abs error {err}"
    return out, ref, kref, vref


@pytest.mark.parametrize("name", ["tiny", "opt13b", "llama8b", "parallel_sampling"])
def test_workload_step(name, kernel):
    w = workloads.make(name, device="cuda")
    out, ref, _, _ = _check_step(w)
    if name == "tiny":
        # fp32 inputs: far tighter than the bar
        assert np.max(np.abs(out.cpu().numpy() - ref)) < 1e-4


@pytest.mark.parametrize("block_size", [8, 16, 32])
def test_long_context_step(block_size, kernel):
    w = workloads.make("long_context", device="cuda", block_size=block_size)
    _check_step(w)


def test_long_context_independent_of_block_size(kernel):
    outs = []
    for bs in (8, 16, 32):
        w = workloads.make("long_context", device="cuda", block_size=bs, num_seqs=2)
        _, _, out, status, _ = gpu_step(w)
        assert status == 0
        outs.append(out)
    assert torch.max(torch.abs(outs[0] - outs[1])) < 1e-5
    assert torch.max(torch.abs(outs[0] - outs[2])) < 1e-5


def test_output_in_query_dtype(kernel):
    w = workloads.make("llama8b", device="cuda", num_seqs=64)
    k, v, out, status, _ = gpu_step(w, out_dtype=torch.bfloat16)
    assert status == 0 and out.dtype == torch.bfloat16
    kref, vref = oracle_pools(w)
    assert max_violation(out, oracle_decode(w, kref, vref)) <= 0.0


@pytest.mark.parametrize("partition", [64, 128, 192, 512, 4096])
def test_forced_partitions(partition, kernel):
    w = workloads.make("llama8b", device="cuda", num_seqs=48)
    _check_step(w, partition_size=partition)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=str)
def test_large_scores(dtype, kernel):
    """A softmax scale 40 times 1/sqrt(d): scores spread over hundreds of
    units, so a row's running max grows many times along the context (every
    rescaling path runs) and the weights are nearly one-hot."""
    w = workloads.custom([1, 40, 300, 777, 2048, 3000], num_heads=32, num_kv_heads=8, head_dim=128,
                         block_size=16, dtype=dtype, num_blocks=None, device="cuda", seed=7400)
    w = dataclasses.replace(w, scale=w.scale * 40.0)
    for partition in (0, 512):
        _check_step(w, partition_size=partition)


LENGTHS = [0, 1, 7, 8, 9, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 129, 200, 513]


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16], ids=str)
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("block_size", [8, 16, 32])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_shape_matrix(dtype, head_dim, block_size, group, kernel):
    w = workloads.custom(LENGTHS, num_heads=2 * group, num_kv_heads=2, head_dim=head_dim, block_size=block_size,
                         dtype=dtype, num_blocks=None, device="cuda",
                         seed=7000 + head_dim + block_size + 10 * group)
    for partition in (0, 64):
        _check_step(w, partition_size=partition)


def test_block_relabelling_invariance(kernel):
    w = workloads.make("llama8b", device="cuda", num_seqs=32)
    _, _, base, status, _ = gpu_step(w)
    assert status == 0
    nb = w.num_blocks
    relabel = torch.randperm(nb, generator=torch.Generator().manual_seed(5)).cuda()
    k = torch.empty_like(w.k_cache)
    v = torch.empty_like(w.v_cache)
    k[relabel] = w.k_cache
    v[relabel] = w.v_cache
    tables = w.block_tables.clone().long()
    used = tables >= 0
    tables[used] = relabel[tables[used]]
    slots = w.slot_mapping
    moved_slots = relabel[slots // w.block_size] * w.block_size + slots % w.block_size
    w2 = workloads.Workload(**{**w.__dict__, "k_cache": k, "v_cache": v, "block_tables": tables.int(),
                               "slot_mapping": moved_slots})
    _, _, again, status, _ = gpu_step(w2)
    assert status == 0
    assert torch.max(torch.abs(base - again)) <= 1e-6


def test_shared_prefix_equals_private_copies(kernel):
    w = workloads.make("parallel_sampling", device="cuda", num_seqs=32)
    _, _, shared, status, _ = gpu_step(w)
    assert status == 0
    # Give every sequence private copies of all its blocks (after the step's
    # copies and writes), then decode again over the unshared pool.
    kref, vref = oracle_pools(w)
    tables = w.block_tables.cpu()
    used = int((tables >= 0).sum())
    k_priv = torch.empty((used,) + tuple(w.k_cache.shape[1:]), dtype=w.dtype)
    v_priv = torch.empty_like(k_priv)
    new_tables = torch.full_like(tables, -1)
    kt = torch.from_numpy(kref).view(w.dtype)
    vt = torch.from_numpy(vref).view(w.dtype)
    nxt = 0
    for s in range(w.num_seqs):
        for j in range(tables.shape[1]):
            b = int(tables[s, j])
            if b < 0:
                continue
            k_priv[nxt] = kt[b]
            v_priv[nxt] = vt[b]
            new_tables[s, j] = nxt
            nxt += 1
    out = api.decode(w.query, k_priv.cuda(), v_priv.cuda(), new_tables.cuda(), w.context_lens, w.scale,
                     max_context_len=w.max_context_len)
    assert torch.max(torch.abs(out - shared)) <= 1e-6


def test_gqa_equals_repeated_mha(kernel):
    """Invariant (5): a GQA step (8 KV heads, 32 query heads) gives what the
    same step gives as MHA with every KV head repeated for its 4 query heads
    (the pools and the new tokens repeated along the head axis)."""
    w = workloads.make("llama8b", device="cuda", num_seqs=24)
    g = w.num_heads // w.num_kv_heads
    mha = dataclasses.replace(
        w, num_kv_heads=w.num_heads,
        k_cache=w.k_cache.repeat_interleave(g, dim=1).contiguous(),
        v_cache=w.v_cache.repeat_interleave(g, dim=1).contiguous(),
        new_key=w.new_key.repeat_interleave(g, dim=1).contiguous(),
        new_value=w.new_value.repeat_interleave(g, dim=1).contiguous())
    _, _, out_gqa, status, code = gpu_step(w, partition_size=512)
    assert (status, code) == (0, 0)
    _, _, out_mha, status, code = gpu_step(mha, partition_size=512)
    assert (status, code) == (0, 0)
    assert torch.max(torch.abs(out_gqa - out_mha)).item() <= 1e-6


def test_copy_blocks_many_layers():
    layers, nb, hkv, bs, d = 3, 64, 4, 16, 128
    g = torch.Generator(device="cuda").manual_seed(11)
    ks = [torch.randn(nb, hkv, bs, d, device="cuda", generator=g).to(torch.bfloat16) for _ in range(layers)]
    vs = [torch.randn(nb, hkv, bs, d, device="cuda", generator=g).to(torch.bfloat16) for _ in range(layers)]
    pairs = torch.tensor([[3, 40], [3, 41], [10, 0], [63, 5]], dtype=torch.int64, device="cuda")
    import oracle as O
    kb = [bits(x).copy() for x in ks]
    vb = [bits(x).copy() for x in vs]
    O.get().copy_blocks(kb, vb, pairs.cpu().numpy())
    api.copy_blocks(ks, vs, pairs)
    assert api.get_device_error() == (0, 0)
    for l in range(layers):
        assert pools_equal(ks[l], kb[l]) and pools_equal(vs[l], vb[l])


def test_negative_slots_are_skipped():
    w = workloads.make("tiny", device="cuda")
    slots = w.slot_mapping.clone()
    slots[1] = -1
    slots[3] = -7
    w2 = workloads.Workload(**{**w.__dict__, "slot_mapping": slots})
    k = w2.k_cache.clone()
    v = w2.v_cache.clone()
    api.reshape_and_cache(w2.new_key, w2.new_value, k, v, slots)
    assert api.get_device_error() == (0, 0)
    kref, vref = oracle_pools(w2)
    assert pools_equal(k, kref) and pools_equal(v, vref)


def test_device_error_block_id():
    w = workloads.make("tiny", device="cuda")
    tables = w.block_tables.clone()
    tables[2, 1] = w.num_blocks + 5
    api.decode(w.query, w.k_cache, w.v_cache, tables, w.context_lens, w.scale, max_context_len=64)
    status, code = api.get_device_error()
    assert status == -5
    assert code & native.DEVERR_BLOCK_ID
    assert api.get_device_error() == (0, 0)  # cleared


def test_device_error_slot_and_pair():
    w = workloads.make("tiny", device="cuda")
    slots = w.slot_mapping.clone()
    slots[0] = w.num_blocks * w.block_size + 3
    k = w.k_cache.clone()
    v = w.v_cache.clone()
    api.reshape_and_cache(w.new_key, w.new_value, k, v, slots)
    status, code = api.get_device_error()
    assert status == -5 and code & native.DEVERR_SLOT
    pairs = torch.tensor([[0, w.num_blocks]], dtype=torch.int64, device="cuda")
    api.copy_blocks([k], [v], pairs)
    status, code = api.get_device_error()
    assert status == -5 and code & native.DEVERR_COPY_PAIR


def test_device_error_context_beyond_hint():
    w = workloads.make("llama8b", device="cuda", num_seqs=8)
    api.decode(w.query, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
               max_context_len=16, partition_size=64)
    status, code = api.get_device_error()
    assert status == -5 and code & native.DEVERR_CONTEXT_LEN


def test_workspace_too_small_is_rejected():
    w = workloads.make("tiny", device="cuda")
    ws = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(native.PaError) as e:
        api.decode(w.query, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale, workspace=ws,
                   max_context_len=64)
    assert e.value.status == -3


def test_repeated_calls_reuse_workspace(kernel):
    w = workloads.make("llama8b", device="cuda", num_seqs=64)
    k, v, first, status, _ = gpu_step(w)
    ws = torch.empty(api.decode_workspace_size(w.num_seqs, w.num_heads, w.max_context_len, 64, w.head_dim),
                     dtype=torch.uint8, device="cuda")
    outs = [api.decode(w.query, k, v, w.block_tables, w.context_lens, w.scale, max_context_len=w.max_context_len,
                       partition_size=64, workspace=ws) for _ in range(3)]
    assert api.get_device_error() == (0, 0)
    for o in outs:
        assert torch.equal(o, outs[0])
    assert torch.max(torch.abs(outs[0] - first)) < ATOL


def test_prepared_decode_matches_decode(kernel):
    """A decode call prepared once and run repeatedly (new contents of the same
    tensors each time) gives what api.decode gives."""
    w = workloads.make("llama8b", device="cuda", num_seqs=48)
    k, v = w.k_cache.clone(), w.v_cache.clone()
    api.reshape_and_cache(w.new_key, w.new_value, k, v, w.slot_mapping)
    mc = int(w.context_lens.max())
    q = w.query.clone()
    out = torch.empty(w.num_seqs, w.num_heads, w.head_dim, device="cuda")
    call = api.PreparedDecode(q, k, v, w.block_tables, w.context_lens, w.scale, out=out, max_context_len=mc,
                              partition_size=512)
    for step in range(3):
        q.copy_(torch.roll(w.query, step, dims=0))  # new queries in the same buffer
        got = call().clone()
        ref = api.decode(q, k, v, w.block_tables, w.context_lens, w.scale, max_context_len=mc, partition_size=512)
        assert api.get_device_error() == (0, 0)
        assert torch.equal(got, ref)


def test_prepared_cache_write_matches_reshape_and_cache():
    """A cache write prepared once and run each step (new token contents and
    slots in the same buffers) leaves the pools bit-identical to
    api.reshape_and_cache."""
    w = workloads.make("llama8b", device="cuda", num_seqs=48)
    k1, v1 = w.k_cache.clone(), w.v_cache.clone()
    k2, v2 = w.k_cache.clone(), w.v_cache.clone()
    key, value, slots = w.new_key.clone(), w.new_value.clone(), w.slot_mapping.clone()
    write = api.PreparedCacheWrite(key, value, k1, v1, slots)
    for step in range(3):
        key.copy_(torch.roll(w.new_key, step, dims=0))
        value.copy_(torch.roll(w.new_value, step, dims=0))
        slots.copy_(torch.roll(w.slot_mapping, step, dims=0))
        write()
        api.reshape_and_cache(key, value, k2, v2, slots)
        assert api.get_device_error() == (0, 0)
        assert torch.equal(k1.view(torch.int16), k2.view(torch.int16))
        assert torch.equal(v1.view(torch.int16), v2.view(torch.int16))


def test_step_captured_in_cuda_graph(kernel):
    """The step's calls can be captured in a CUDA graph (no allocation, no
    synchronisation inside them) and the replay gives the same outputs."""
    w = workloads.make("llama8b", device="cuda", num_seqs=32)
    mc = int(w.context_lens.max())
    k, v = w.k_cache.clone(), w.v_cache.clone()
    ws = torch.empty(api.decode_workspace_size(w.num_seqs, w.num_heads, mc, 0, w.head_dim), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty(w.num_seqs, w.num_heads, w.head_dim, device="cuda")

    def step():
        api.reshape_and_cache(w.new_key, w.new_value, k, v, w.slot_mapping)
        api.decode(w.query, k, v, w.block_tables, w.context_lens, w.scale, out=out, max_context_len=mc,
                   workspace=ws)

    step()
    torch.cuda.synchronize()
    ref = out.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            step()
    out.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert api.get_device_error() == (0, 0)
    assert torch.equal(out, ref)


def test_many_sequences():
    """3000 sequences: the planning kernel's scan spans several 1024-sequence
    chunks, and the decode kernel several waves of work items."""
    g = torch.Generator().manual_seed(31)
    lens = torch.randint(0, 700, (3000,), generator=g).tolist()
    w = workloads.custom(lens, num_heads=8, num_kv_heads=2, head_dim=64, block_size=16, dtype=torch.bfloat16,
                         device="cuda", seed=313)
    for partition in (0, 128):
        _check_step(w, partition_size=partition)


def test_longest_context():
    """One 131072-token sequence next to short ones (256 partitions of 512)."""
    w = workloads.custom([131072, 3, 700], num_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                         dtype=torch.bfloat16, device="cuda", seed=314)
    _check_step(w, partition_size=512)


def test_beam_search_trace(kernel):
    """Beam search with forks, deaths and copy-on-write at every step: the
    pools match the oracle bit for bit after every step, and every step's
    attention matches within the bar."""
    import oracle as O

    t = workloads.beam_search(beams=4, prompt_len=45, steps=40, block_size=8, num_heads=8, num_kv_heads=2,
                              head_dim=64, dtype=torch.bfloat16, device="cuda")
    assert sum(st.copy_pairs.shape[0] for st in t.steps) > 0
    orc = O.get()
    k, v = t.k_cache.clone(), t.v_cache.clone()
    kb, vb = bits(t.k_cache).copy(), bits(t.v_cache).copy()
    for st in t.steps:
        if st.copy_pairs.numel():
            api.copy_blocks([k], [v], st.copy_pairs)
            orc.copy_blocks([kb], [vb], st.copy_pairs.cpu().numpy())
        api.reshape_and_cache(st.new_key, st.new_value, k, v, st.slot_mapping)
        orc.reshape_and_cache(bits(st.new_key), bits(st.new_value), kb, vb, st.slot_mapping.cpu().numpy())
        out = api.decode(st.query, k, v, st.block_tables, st.context_lens, t.scale,
                         max_context_len=int(st.context_lens.max()))
        assert api.get_device_error() == (0, 0)
        assert pools_equal(k, kb) and pools_equal(v, vb)
        ref = orc.decode(bits(st.query), kb, vb, O.BF16, st.block_tables.cpu().numpy(),
                         st.context_lens.cpu().numpy(), t.num_kv_heads, t.scale)
        assert max_violation(out, ref) <= 0.0


@pytest.mark.parametrize("partition,max_len", [(64, 700), (0, 700), (512, 512)])
def test_many_sequences_each_kernel(partition, max_len, kernel):
    """3000 sequences with both decode kernels: at partition 64 the reduce
    kernel strides over more (sequence, head) pairs than its grid has warps,
    and with every context inside one partition the items map to CTAs
    directly, many per CTA."""
    g = torch.Generator().manual_seed(3000 + partition)
    lens = torch.randint(1, max_len + 1, (3000,), generator=g).tolist()
    w = workloads.custom(lens, num_heads=8, num_kv_heads=2, head_dim=64, block_size=16, dtype=torch.bfloat16,
                         device="cuda", seed=3100 + partition)
    _check_step(w, partition_size=partition)
