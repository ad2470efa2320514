"""Head-sharded decode on one GPU ("PagedAttention 论文精读笔记", §8.1 and §8.2).

The pools are sliced by KV head into N shards that keep the block ids; each
shard runs the step (copy-on-write, cache write, decode) through the C ABI
with the same tables, slots and partition size.  The shards' outputs,
concatenated along the head axis, must equal the unsharded call bit for bit
(each (sequence, KV head) item is computed the same way whatever the other
heads are), and be within the 2e-3 bar of the oracle.  The shards' pools must
equal the matching heads of the unsharded pools bit for bit.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_132_gb300 import native, sharding, workloads
from steps import bits, gpu_step, max_violation, oracle_decode, oracle_pools

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    native.load()


@pytest.mark.parametrize("name,kw,partition,worlds", [
    ("llama8b", {"num_seqs": 64}, 512, (2, 4, 8)),
    ("opt13b", {"num_seqs": 16}, 512, (2, 4, 5)),
    ("parallel_sampling", {}, 512, (2, 4)),
    ("long_context", {"num_seqs": 2, "block_size": 16}, 512, (2, 8)),
    ("tiny", {}, 64, (2, 4)),
])
def test_shards_concatenate_to_the_unsharded_call(name, kw, partition, worlds):
    w = workloads.make(name, device="cuda", **kw)
    k_full, v_full, full, status, code = gpu_step(w, partition_size=partition)
    assert (status, code) == (0, 0)
    kref, vref = oracle_pools(w)
    ref = oracle_decode(w, kref, vref)
    assert max_violation(full, ref) <= 0.0
    for world in worlds:
        outs = []
        for r in range(world):
            shard = sharding.shard_workload(w, world, r)
            k, v, out, status, code = gpu_step(shard, partition_size=partition)
            assert (status, code) == (0, 0), f"{world} shards, rank {r}: device error {status} / {code:#x}"
            assert np.array_equal(bits(k), bits(sharding.shard_pool(k_full, world, r))), "K shard differs"
            assert np.array_equal(bits(v), bits(sharding.shard_pool(v_full, world, r))), "V shard differs"
            outs.append(out)
        got = sharding.concat_heads(outs)
        assert torch.equal(got, full), f"{name}: {world} shards differ from the unsharded call"
        assert max_violation(got, ref) <= 0.0
