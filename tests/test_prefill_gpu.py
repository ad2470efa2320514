"""GPU parity of the prefill over a cached prefix (tensor cores) against the
fp64 oracle.

A step is: copy-on-write of the shared partial prefix block, the cache write
of the new tokens, then pa_prefill.  Pools must match the oracle bit for bit;
attention outputs within 2e-3 absolute (plus half an ulp of a 16-bit output
type).  Every slot that holds no cached token is NaN.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
from paged_kv_cache_132_gb300 import api, native, workloads
from steps import CODE, bits, max_violation, pools_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    native.load()


def gpu_prefill_step(st, out_dtype=torch.float32, max_query_len=None, extra_rows=0):
    k = st.k_cache.clone()
    v = st.v_cache.clone()
    if st.copy_pairs.numel():
        api.copy_blocks([k], [v], st.copy_pairs)
    api.reshape_and_cache(st.new_key, st.new_value, k, v, st.slot_mapping)
    query = st.query
    out = None
    if extra_rows:
        # rows after the last sequence's: not read for any output, never written
        query = torch.cat([st.query, torch.randn(extra_rows, *st.query.shape[1:], device="cuda").to(st.dtype)])
        out = torch.full((query.shape[0], st.num_heads, st.head_dim), 7.0, dtype=out_dtype, device="cuda")
    out = api.prefill(query, st.query_start_loc, k, v, st.block_tables, st.context_lens, st.scale,
                      st.max_query_len if max_query_len is None else max_query_len, out=out, out_dtype=out_dtype)
    status, code = api.get_device_error()
    return k, v, out, status, code


def oracle_step_pools(st):
    orc = O.get()
    k = bits(st.k_cache).copy()
    v = bits(st.v_cache).copy()
    if st.copy_pairs.numel():
        orc.copy_blocks([k], [v], st.copy_pairs.cpu().numpy())
    orc.reshape_and_cache(bits(st.new_key), bits(st.new_value), k, v, st.slot_mapping.cpu().numpy())
    return k, v


def oracle_prefill(st, k_bits, v_bits, seqs=None):
    """fp64 outputs [rows][H][d] of all sequences, or of the listed ones (their
    rows in list order)."""
    orc = O.get()
    qsl = st.query_start_loc.cpu().numpy()
    tables = st.block_tables.cpu().numpy()
    ctx = st.context_lens.cpu().numpy()
    q = st.query.cpu()
    if seqs is not None:
        rows = np.concatenate([np.arange(qsl[s], qsl[s + 1]) for s in seqs])
        lens = [qsl[s + 1] - qsl[s] for s in seqs]
        qsl = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        q = q[torch.as_tensor(rows, dtype=torch.int64)]
        tables = tables[np.asarray(seqs)]
        ctx = ctx[np.asarray(seqs)]
    return orc.prefill(bits(q), qsl, k_bits, v_bits, CODE[st.dtype], tables, ctx, st.num_kv_heads, st.scale,
                       num_threads=0)


def check(st, **kw):
    k, v, out, status, code = gpu_prefill_step(st, **kw)
    assert status == 0 and code == 0, f"device error {status} / {code:#x}"
    kref, vref = oracle_step_pools(st)
    assert pools_equal(k, kref) and pools_equal(v, vref), "pools differ from the oracle"
    ref = oracle_prefill(st, kref, vref)
    got = out[: st.num_tokens]
    err = float(np.max(np.abs(got.float().cpu().numpy() - ref))) if ref.size else 0.0
    assert max_violation(got, ref) <= 0.0, f"max abs error {err}"
    return out, ref, err


def test_prefill_tiny():
    st = workloads.make_prefill("prefill_tiny", device="cuda")
    _, _, err = check(st)
    assert err < 2e-3


SHAPES = [
    # (dtype, head_dim, heads, kv_heads, block_size)
    (torch.bfloat16, 128, 32, 8, 16),
    (torch.bfloat16, 128, 8, 8, 32),
    (torch.bfloat16, 64, 16, 8, 8),
    (torch.bfloat16, 64, 8, 1, 16),
    (torch.float16, 128, 40, 40, 16),
    (torch.float16, 128, 16, 2, 8),
    (torch.float16, 64, 4, 2, 32),
    (torch.float16, 64, 32, 4, 16),
]


@pytest.mark.parametrize("dtype,d,h,hkv,bs", SHAPES)
def test_prefill_shapes(dtype, d, h, hkv, bs):
    # chunks: 1 token, ragged tiles, several query tiles; prefixes: none,
    # unaligned, several key tiles long; an empty chunk in the middle
    st = workloads.prefill_custom([1, 77, 0, 300, 129], [0, 45, 333], prefix_groups=[1, 0, 2, 1, 2],
                                  num_heads=h, num_kv_heads=hkv, head_dim=d, block_size=bs, dtype=dtype,
                                  seed=7100 + d + h + bs, device="cuda")
    check(st)


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float16, 128), (torch.bfloat16, 64)])
def test_prefill_large_scores(dtype, d):
    """A softmax scale 40 times 1/sqrt(d): a row's running max grows many
    times along the keys (the rescaling of O, and of P inside a tile, runs)
    and the weights are nearly one-hot."""
    st = workloads.prefill_custom([1, 77, 300, 129], [0, 45, 1000], prefix_groups=[1, 0, 2, 2],
                                  num_heads=16, num_kv_heads=4, head_dim=d, block_size=16, dtype=dtype,
                                  seed=7500 + d, device="cuda")
    check(dataclasses.replace(st, scale=st.scale * 40.0))


@pytest.mark.parametrize("out_dtype", [torch.float16, torch.bfloat16])
def test_prefill_output_dtypes(out_dtype):
    st = workloads.make_prefill("prefill_tiny", device="cuda")
    check(st, out_dtype=out_dtype)


def test_prefill_rows_outside_sequences_untouched():
    st = workloads.make_prefill("prefill_tiny", device="cuda")
    out, _, _ = check(st, extra_rows=40, max_query_len=200)
    assert torch.all(out[st.num_tokens:] == 7.0)


def test_prefill_one_token_chunks_match_decode():
    # n = 1 for every sequence: prefill is the decode step
    st = workloads.prefill_custom([1] * 6, [900, 17, 128, 1, 2000, 64], num_heads=32, num_kv_heads=8,
                                  head_dim=128, block_size=16, dtype=torch.bfloat16, seed=7200, device="cuda")
    k, v, out, status, code = gpu_prefill_step(st)
    assert status == 0 and code == 0
    dec = api.decode(st.query, k, v, st.block_tables, st.context_lens, st.scale, max_context_len=2001)
    assert float((out - dec).abs().max()) < 2e-3


def test_prefill_long_shared_prefix():
    # 8 requests share a 6000-token prefix; chunks span many query tiles
    st = workloads.prefill_custom([700, 1, 513, 64, 1000, 255, 129, 4], [6000], prefix_groups=[0] * 8,
                                  num_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                                  dtype=torch.bfloat16, seed=7300, device="cuda")
    k, v, out, status, code = gpu_prefill_step(st)
    assert status == 0 and code == 0
    kref, vref = oracle_step_pools(st)
    seqs = [1, 3, 6, 7]
    ref = oracle_prefill(st, kref, vref, seqs)
    qsl = st.query_start_loc.cpu().numpy()
    rows = np.concatenate([np.arange(qsl[s], qsl[s + 1]) for s in seqs])
    got = out[torch.as_tensor(rows, device="cuda")]
    assert max_violation(got, ref) <= 0.0


@pytest.mark.parametrize("name", ["prefill_llama8b", "prefill_opt13b"])
def test_prefill_full_size_sampled(name):
    """The bench's workloads at full size, compared on sampled sequences (the
    oracle computes those in seconds); every output must be finite."""
    st = workloads.make_prefill(name, device="cuda")
    k, v, out, status, code = gpu_prefill_step(st)
    assert status == 0 and code == 0
    assert bool(torch.isfinite(out).all())
    kref, vref = oracle_step_pools(st)
    assert pools_equal(k, kref) and pools_equal(v, vref)
    seqs = [0, st.num_seqs // 2, st.num_seqs - 1]
    ref = oracle_prefill(st, kref, vref, seqs)
    qsl = st.query_start_loc.cpu().numpy()
    rows = np.concatenate([np.arange(qsl[s], qsl[s + 1]) for s in seqs])
    got = out[torch.as_tensor(rows, device="cuda")]
    assert max_violation(got, ref) <= 0.0


def test_prefill_grid_order_for_pools_larger_than_l2():
    """Pools above the L2 size switch the grid to keep each (sequence, KV
    head)'s query tiles together; every CTA computes the same tile either
    way, so the outputs are bit-identical.  The same step is run on its own
    pools and on the pools padded with unused (NaN) blocks past L2's size."""
    st = workloads.make_prefill("prefill_tiny", device="cuda")
    k, v, out, status, _ = gpu_prefill_step(st)
    assert status == 0
    block_bytes = k[0].numel() * k.element_size()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    pad = (l2 // block_bytes) // 2 + 1  # K and V together exceed L2
    kp = torch.cat([k, torch.full((pad,) + tuple(k.shape[1:]), float("nan"), dtype=k.dtype, device="cuda")])
    vp = torch.cat([v, torch.full((pad,) + tuple(v.shape[1:]), float("nan"), dtype=v.dtype, device="cuda")])
    assert 2 * kp.numel() * kp.element_size() > l2
    out2 = api.prefill(st.query, st.query_start_loc, kp, vp, st.block_tables, st.context_lens, st.scale,
                       st.max_query_len)
    assert api.get_device_error() == (0, 0)
    assert torch.equal(out, out2)


def test_prefill_relabelled_blocks_identical():
    """Moving every block to another physical id (and fixing the tables)
    leaves every output bit unchanged."""
    st = workloads.make_prefill("prefill_tiny", device="cuda")
    k, v, out, status, _ = gpu_prefill_step(st)
    assert status == 0
    perm = torch.randperm(st.num_blocks, generator=torch.Generator().manual_seed(5)).cuda()
    k2 = torch.empty_like(k)
    v2 = torch.empty_like(v)
    k2[perm] = k
    v2[perm] = v
    tables = st.block_tables.clone()
    mask = tables >= 0
    tables[mask] = perm[tables[mask].long()].int()
    out2 = api.prefill(st.query, st.query_start_loc, k2, v2, tables, st.context_lens, st.scale, st.max_query_len)
    assert torch.equal(out, out2)


def test_prefill_bad_lengths_reported():
    """A chunk longer than its context is refused by the kernel (the
    sequence is skipped, PA_DEVERR_CONTEXT_LEN); the others are computed."""
    st = workloads.make_prefill("prefill_tiny", device="cuda")
    k, v, out, status, code = gpu_prefill_step(st)
    bad_ctx = st.context_lens.clone()
    bad_ctx[1] = 10  # chunk of 50 tokens
    out2 = torch.full_like(out, 3.0)
    api.prefill(st.query, st.query_start_loc, k, v, st.block_tables, bad_ctx, st.scale, st.max_query_len,
                out=out2)
    status, code = api.get_device_error()
    assert status == -5 and code & native.DEVERR_CONTEXT_LEN
    qsl = st.query_start_loc.cpu().tolist()
    assert torch.all(out2[qsl[1]:qsl[2]] == 3.0)
    assert torch.equal(out2[: qsl[1]], out[: qsl[1]]) and torch.equal(out2[qsl[2]:], out[qsl[2]:])
