"""pa_swap_blocks: blocks between a GPU pool and a page-locked host pool.

Swapping ("PagedAttention 论文精读笔记", §7.4) copies a preempted sequence's
blocks to CPU memory and back into (possibly other) GPU blocks when it
resumes.  Checks: bit-exact against the oracle in both directions over the
whole destination pool, attention unchanged after a swap-out / swap-in round
trip into different blocks, rejected pageable memory, out-of-range pairs.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
from paged_kv_cache_132_gb300 import api, native, workloads
from steps import bits, gpu_step, pools_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    assert torch.cuda.is_available()
    native.load()


def _host_pool(like, blocks, fill=float("nan")):
    return torch.full((blocks,) + tuple(like.shape[1:]), fill, dtype=like.dtype).pin_memory()


@pytest.mark.parametrize("layers", [1, 2])
def test_swap_out_and_in_bit_exact(layers):
    g = torch.Generator(device="cuda").manual_seed(21)
    nb, host_nb, shape = 300, 120, (8, 16, 128)
    gk = [torch.randn((nb,) + shape, generator=g, device="cuda").to(torch.bfloat16) for _ in range(layers)]
    gv = [torch.randn((nb,) + shape, generator=g, device="cuda").to(torch.bfloat16) for _ in range(layers)]
    hk = [_host_pool(gk[0], host_nb) for _ in range(layers)]
    hv = [_host_pool(gk[0], host_nb) for _ in range(layers)]
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(3))
    out_pairs = torch.stack([perm[:100], torch.randperm(host_nb, generator=torch.Generator().manual_seed(4))[:100]],
                            dim=1).contiguous().cuda()
    ref_hk = [bits(x).copy() for x in hk]
    ref_hv = [bits(x).copy() for x in hv]
    O.get().swap_blocks([bits(x) for x in gk], [bits(x) for x in gv], ref_hk, ref_hv, out_pairs.cpu().numpy())
    api.swap_blocks(gk, gv, hk, hv, out_pairs)
    assert api.get_device_error() == (0, 0)
    for l in range(layers):
        assert np.array_equal(bits(hk[l]), ref_hk[l]) and np.array_equal(bits(hv[l]), ref_hv[l])
    # swap-in into other GPU blocks (pairs given in pinned host memory)
    in_pairs = torch.stack([out_pairs[:, 1].cpu(), perm[200:300]], dim=1).contiguous().pin_memory()
    ref_gk = [bits(x).copy() for x in gk]
    ref_gv = [bits(x).copy() for x in gv]
    O.get().swap_blocks([bits(x) for x in hk], [bits(x) for x in hv], ref_gk, ref_gv, in_pairs.numpy())
    api.swap_blocks(hk, hv, gk, gv, in_pairs)
    assert api.get_device_error() == (0, 0)
    for l in range(layers):
        assert pools_equal(gk[l], ref_gk[l]) and pools_equal(gv[l], ref_gv[l])


def test_swap_round_trip_keeps_attention():
    w = workloads.make("llama8b", device="cuda", num_seqs=32)
    k, v, base, status, _ = gpu_step(w)
    assert status == 0
    victims = list(range(8))  # preempt sequences 0..7
    tables = w.block_tables.clone()
    blocks = sorted({int(b) for s in victims for b in tables[s].tolist() if b >= 0})
    hk, hv = _host_pool(k, len(blocks)), _host_pool(v, len(blocks))
    out_pairs = torch.tensor([[b, i] for i, b in enumerate(blocks)], dtype=torch.int64, device="cuda")
    api.swap_blocks([k], [v], [hk], [hv], out_pairs)
    # their GPU blocks are reused by someone else meanwhile
    k[torch.tensor(blocks, device="cuda")] = float("nan")
    v[torch.tensor(blocks, device="cuda")] = float("nan")
    # resume into a larger pool, at fresh block ids
    extra = len(blocks)
    k2 = torch.cat([k, torch.full((extra,) + tuple(k.shape[1:]), float("nan"), dtype=k.dtype, device="cuda")])
    v2 = torch.cat([v, torch.full_like(k2[-extra:], float("nan"))])
    new_ids = list(range(w.num_blocks, w.num_blocks + extra))
    in_pairs = torch.tensor([[i, new_ids[i]] for i in range(extra)], dtype=torch.int64, device="cuda")
    api.swap_blocks([hk], [hv], [k2], [v2], in_pairs)
    remap = {b: new_ids[i] for i, b in enumerate(blocks)}
    for s in victims:
        for j in range(tables.shape[1]):
            b = int(tables[s, j])
            if b >= 0:
                tables[s, j] = remap[b]
    out = api.decode(w.query, k2, v2, tables, w.context_lens, w.scale, max_context_len=int(w.context_lens.max()))
    assert api.get_device_error() == (0, 0)
    assert torch.max(torch.abs(out - base)).item() <= 1e-6


def test_swap_rejects_pageable_memory_and_bad_pairs():
    nb, shape = 16, (2, 8, 64)
    gk = torch.zeros((nb,) + shape, dtype=torch.float16, device="cuda")
    gv = torch.zeros_like(gk)
    pageable = np.zeros((nb,) + shape, dtype=np.float16)
    pairs = torch.tensor([[0, 1]], dtype=torch.int64, device="cuda")
    desc = api.cache_desc(gk)
    P = ctypes.c_void_p * 1
    status = native.load().pa_swap_blocks(P(gk.data_ptr()), P(gv.data_ptr()), nb, P(pageable.ctypes.data),
                                          P(pageable.ctypes.data), nb, 1, pairs.data_ptr(), 1, ctypes.byref(desc),
                                          None)
    assert status == -1  # PA_ERR_INVALID_ARG: the GPU cannot address pageable host memory here
    hk = _host_pool(gk, 4, 0.0)
    hv = _host_pool(gk, 4, 0.0)
    bad = torch.tensor([[0, 4]], dtype=torch.int64, device="cuda")  # host pool has 4 blocks
    api.swap_blocks([gk], [gv], [hk], [hv], bad)
    status, code = api.get_device_error()
    assert status == -5 and code & native.DEVERR_COPY_PAIR
