"""Randomised steps against the oracle.

The shape matrix of the other parity tests walks each axis on its own; here
every case draws all of them at once from the supported space -- pool dtype,
head_dim, block size, KV heads, GQA group, output dtype, split-KV partition,
batch size and context lengths (edge lengths around block and partition
boundaries mixed with random ones) -- and checks one step: the pools bit for
bit after the cache write, attention within the bar on every output.  The
prefill cases draw chunk and prefix lengths the same way.  Seeds are fixed,
so a failure names a reproducible case.
"""
import random

import pytest
import torch

import oracle as O
from paged_kv_cache_132_gb300 import api, native, workloads
from steps import CODE, bits, gpu_step, max_violation, oracle_decode, oracle_pools, pools_equal

pytestmark = pytest.mark.gpu

DTYPES = [torch.float32, torch.float16, torch.bfloat16]


@pytest.fixture(scope="module", autouse=True)
def _library():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    native.load()


def _lengths(rng, n, block_size, part):
    edges = [0, 1, block_size - 1, block_size, block_size + 1, 63, 64, 65]
    if part:
        edges += [part - 1, part, part + 1, 2 * part + 3]
    return [rng.choice(edges) if rng.random() < 0.4 else rng.randint(1, 2500) for _ in range(n)]


def _decode_case(seed):
    rng = random.Random(9000 + seed)
    dtype = rng.choice(DTYPES)
    d = rng.choice([64, 128])
    bs = rng.choice([8, 16, 32])
    hkv = rng.choice([1, 2, 4, 8])
    group = rng.choice([1, 2, 4, 8])
    part = rng.choice([0, 64, 128, 512, 1024])
    out_dtype = rng.choice([torch.float32, dtype])
    ctx = _lengths(rng, rng.randint(1, 24), bs, part)
    return dict(ctx=ctx, num_heads=hkv * group, num_kv_heads=hkv, head_dim=d, block_size=bs, dtype=dtype,
                partition_size=part), out_dtype


@pytest.mark.parametrize("seed", range(64))
def test_random_decode_step(seed):
    spec, out_dtype = _decode_case(seed)
    w = workloads.custom(spec.pop("ctx"), **spec, seed=workloads.SEED_BASE + 700 + seed, device="cuda")
    k, v, out, status, code = gpu_step(w, out_dtype=out_dtype)
    assert (status, code) == (0, 0), (seed, spec)
    kref, vref = oracle_pools(w)
    assert pools_equal(k, kref) and pools_equal(v, vref), (seed, spec)
    ref = oracle_decode(w, kref, vref)
    assert max_violation(out, ref) <= 0.0, (seed, spec, out_dtype)


@pytest.mark.parametrize("seed", range(24))
def test_random_prefill_step(seed):
    rng = random.Random(9100 + seed)
    dtype = rng.choice([torch.float16, torch.bfloat16])
    d = rng.choice([64, 128])
    bs = rng.choice([8, 16, 32])
    hkv = rng.choice([1, 2, 4])
    group = rng.choice([1, 2, 4, 8])
    n = rng.randint(1, 6)
    chunks = [rng.choice([0, 1, 31, 32, 33, 127, 128, 129]) if rng.random() < 0.4 else rng.randint(1, 400)
              for _ in range(n)]
    prefixes = [rng.choice([0, bs - 1, bs, 63, 64, 65, rng.randint(1, 700)]) for _ in range(rng.randint(1, 3))]
    groups = [rng.randrange(len(prefixes)) for _ in range(n)]
    st = workloads.prefill_custom(chunks, prefixes, prefix_groups=groups, num_heads=hkv * group, num_kv_heads=hkv,
                                  head_dim=d, block_size=bs, dtype=dtype, seed=workloads.SEED_BASE + 800 + seed,
                                  device="cuda")
    out_dtype = rng.choice([torch.float32, dtype])
    k, v = st.k_cache.clone(), st.v_cache.clone()
    if st.copy_pairs.numel():
        api.copy_blocks([k], [v], st.copy_pairs)
    api.reshape_and_cache(st.new_key, st.new_value, k, v, st.slot_mapping)
    out = api.prefill(st.query, st.query_start_loc, k, v, st.block_tables, st.context_lens, st.scale,
                      st.max_query_len, out_dtype=out_dtype)
    assert api.get_device_error() == (0, 0), (seed, chunks, prefixes)
    orc = O.get()
    kref, vref = bits(st.k_cache).copy(), bits(st.v_cache).copy()
    if st.copy_pairs.numel():
        orc.copy_blocks([kref], [vref], st.copy_pairs.cpu().numpy())
    orc.reshape_and_cache(bits(st.new_key), bits(st.new_value), kref, vref, st.slot_mapping.cpu().numpy())
    assert pools_equal(k, kref) and pools_equal(v, vref), (seed, chunks, prefixes)
    ref = orc.prefill(bits(st.query.cpu()), st.query_start_loc.cpu().numpy(), kref, vref, CODE[st.dtype],
                      st.block_tables.cpu().numpy(), st.context_lens.cpu().numpy(), st.num_kv_heads, st.scale,
                      num_threads=0)
    assert max_violation(out[: st.num_tokens], ref) <= 0.0, (seed, chunks, prefixes, out_dtype)
