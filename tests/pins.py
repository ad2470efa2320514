"""Checks that pin the CPU oracle to facts outside itself.

Each ``check_*`` takes an oracle instance and raises AssertionError when the
oracle disagrees with: a library routine on a special case (torch float64
scaled_dot_product_attention, numpy/torch float conversion), a closed form,
an invariant of paging, or a worked example printed on the pages (fixtures in
``tests/golden/page_examples.json``, each with its citation).  The same checks
run against deliberately broken copies of the oracle in
``test_oracle_mutants.py``, where at least one of them must fail.
"""
from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as F

import oracle as O
from paged_kv_cache_132_gb300 import metrics
from paged_kv_cache_132_gb300.block_manager import BlockManager, blocks_needed, wasted_slots

TORCH_OF = {O.F32: torch.float32, O.F16: torch.float16, O.BF16: torch.bfloat16}


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw element bits of a CPU tensor, in the form the oracle takes."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.float32:
        return t.numpy()
    return t.view(torch.int16).numpy()


def code_of(dtype: torch.dtype) -> int:
    return {torch.float32: O.F32, torch.float16: O.F16, torch.bfloat16: O.BF16}[dtype]


# ---------------------------------------------------------------------------
# a paged case built from contiguous per-sequence K/V
# ---------------------------------------------------------------------------
def paged_case(seed, lens, num_heads, num_kv_heads, head_dim, block_size, dtype_code,
               extra_blocks=3, stale="nan"):
    g = torch.Generator().manual_seed(seed)
    tdt = TORCH_OF[dtype_code]
    s = len(lens)
    nblk = [blocks_needed(n, block_size) for n in lens]
    nb = sum(nblk) + extra_blocks
    perm = torch.randperm(nb, generator=g).tolist()
    tables = np.full((s, max(max(nblk + [0]), 1)), -1, dtype=np.int32)
    cursor = 0
    for i, n in enumerate(nblk):
        tables[i, :n] = perm[cursor: cursor + n]
        cursor += n
    keys = [torch.randn(n, num_kv_heads, head_dim, generator=g).to(tdt) for n in lens]
    values = [torch.randn(n, num_kv_heads, head_dim, generator=g).to(tdt) for n in lens]
    query = torch.randn(s, num_heads, head_dim, generator=g).to(tdt)
    if stale == "nan":
        kp = torch.full((nb, num_kv_heads, block_size, head_dim), float("nan"), dtype=tdt)
        vp = kp.clone()
    else:
        kp = torch.randn(nb, num_kv_heads, block_size, head_dim, generator=g).to(tdt)
        vp = torch.randn(nb, num_kv_heads, block_size, head_dim, generator=g).to(tdt)
    for i, n in enumerate(lens):
        for j in range(n):
            kp[tables[i, j // block_size], :, j % block_size, :] = keys[i][j]
            vp[tables[i, j // block_size], :, j % block_size, :] = values[i][j]
    return dict(lens=list(lens), H=num_heads, Hkv=num_kv_heads, d=head_dim, B=block_size,
                code=dtype_code, tables=tables, keys=keys, values=values, query=query,
                k_pool=kp, v_pool=vp, scale=1.0 / math.sqrt(head_dim))


def run_decode(orc, case, **kw):
    return orc.decode(bits(case["query"]), bits(case["k_pool"]), bits(case["v_pool"]), case["code"],
                      case["tables"], np.array(case["lens"], dtype=np.int32), case["Hkv"],
                      case["scale"], **kw)


def sdpa_reference(case):
    """torch float64 scaled_dot_product_attention on each sequence's contiguous K/V."""
    outs = []
    for i, n in enumerate(case["lens"]):
        q = case["query"][i].to(torch.float64)[None, :, None, :]          # [1, H, 1, d]
        k = case["keys"][i].to(torch.float64).permute(1, 0, 2)[None]      # [1, Hkv, n, d]
        v = case["values"][i].to(torch.float64).permute(1, 0, 2)[None]
        o = F.scaled_dot_product_attention(q, k, v, scale=case["scale"],
                                           enable_gqa=case["H"] != case["Hkv"])
        outs.append(o[0, :, 0, :].numpy())
    return np.stack(outs)


SDPA_CASES = [
    # (lens, H, Hkv, d, B, dtype)
    ([5, 17, 33, 64], 4, 4, 64, 16, O.F32),
    ([1, 2, 9, 40, 16], 8, 2, 32, 8, O.BF16),
    ([3, 31, 32, 33, 70], 6, 3, 16, 4, O.F16),
    ([100, 7], 16, 4, 128, 32, O.BF16),
]


def check_sdpa(orc):
    for idx, (lens, h, hkv, d, b, code) in enumerate(SDPA_CASES):
        case = paged_case(500 + idx, lens, h, hkv, d, b, code)
        got = run_decode(orc, case)
        ref = sdpa_reference(case)
        err = float(np.max(np.abs(got - ref)))
        assert err <= 1e-12, f"oracle vs torch SDPA (case {idx}): max err {err}"


def check_weight_sums(orc):
    case = paged_case(601, [1, 5, 37], 4, 2, 32, 8, O.BF16)
    _, wsum = run_decode(orc, case, want_weight_sum=True)
    assert np.all(np.abs(wsum - 1.0) <= 1e-12), f"weight sums {wsum}"


def check_block_permutation(orc):
    case = paged_case(602, [13, 40, 7], 4, 2, 16, 4, O.F16)
    base = run_decode(orc, case)
    nb = case["k_pool"].shape[0]
    relabel = torch.randperm(nb, generator=torch.Generator().manual_seed(9)).numpy()
    moved = dict(case)
    kp = torch.empty_like(case["k_pool"])
    vp = torch.empty_like(case["v_pool"])
    kp[torch.from_numpy(relabel)] = case["k_pool"]
    vp[torch.from_numpy(relabel)] = case["v_pool"]
    tables = case["tables"].copy()
    used = tables >= 0
    tables[used] = relabel[tables[used]]
    moved.update(k_pool=kp, v_pool=vp, tables=tables)
    again = run_decode(orc, moved)
    assert np.array_equal(base, again), "output changed under a relabelling of physical blocks"


def check_stale_slots_ignored(orc):
    nan_case = paged_case(603, [3, 18, 30], 4, 4, 16, 8, O.BF16, stale="nan")
    rnd_case = paged_case(603, [3, 18, 30], 4, 4, 16, 8, O.BF16, stale="random")
    a = run_decode(orc, nan_case)
    b = run_decode(orc, rnd_case)
    assert np.all(np.isfinite(a)), "a NaN-poisoned stale slot reached the output"
    assert np.array_equal(a, b), "stale-slot contents changed the output"


def check_gqa_equals_repeated_mha(orc):
    case = paged_case(604, [9, 26], 8, 2, 16, 4, O.F32)
    gqa = run_decode(orc, case)
    g = case["H"] // case["Hkv"]
    mha = dict(case)
    mha.update(Hkv=case["H"], k_pool=case["k_pool"].repeat_interleave(g, dim=1).contiguous(),
               v_pool=case["v_pool"].repeat_interleave(g, dim=1).contiguous())
    out = run_decode(orc, mha)
    assert np.array_equal(gqa, out), "GQA differs from MHA with each KV head repeated G times"


def check_closed_forms(orc):
    # (a) all keys equal: uniform weights, output = mean of the values.
    case = paged_case(605, [11], 2, 1, 8, 4, O.F32)
    case["k_pool"][:] = 0.25
    got = run_decode(orc, case)
    mean = case["values"][0].to(torch.float64).mean(dim=0)[0].numpy()
    assert np.max(np.abs(got[0] - mean[None, :])) <= 1e-12, "equal keys must average V"
    # (b) one dominant score: output = that token's value.
    case = paged_case(606, [12], 1, 1, 8, 4, O.F32)
    q = case["query"][0, 0]
    j = 7
    tables = case["tables"]
    case["k_pool"][tables[0, j // 4], 0, j % 4, :] = q * 1000.0
    got = run_decode(orc, case)
    vj = case["values"][0][j, 0].to(torch.float64).numpy()
    assert np.max(np.abs(got[0, 0] - vj)) <= 1e-12, "a dominant score must select its value"
    # (c) one token: output = v_0 exactly.
    case = paged_case(607, [1, 1], 4, 2, 16, 8, O.BF16)
    got = run_decode(orc, case)
    for i in range(2):
        v0 = case["values"][i][0].to(torch.float64).numpy()  # [Hkv][d]
        assert np.array_equal(got[i], np.repeat(v0, 2, axis=0)), "ctx = 1 must return v_0 exactly"
    # (d) no tokens: output 0, weight sum 0.
    case = paged_case(608, [0, 4], 2, 2, 8, 4, O.F16)
    got, wsum = run_decode(orc, case, want_weight_sum=True)
    assert np.all(got[0] == 0.0) and np.all(wsum[0] == 0.0), "ctx = 0 must give zeros"


def check_partition_merge(orc):
    case = paged_case(609, [1, 15, 16, 17, 100, 257], 4, 2, 16, 8, O.BF16)
    single = run_decode(orc, case)
    for part in (1, 3, 16, 64, 1000):
        merged = orc.decode_partitioned(bits(case["query"]), bits(case["k_pool"]),
                                        bits(case["v_pool"]), case["code"], case["tables"],
                                        np.array(case["lens"], dtype=np.int32), case["Hkv"],
                                        case["scale"], part)
        err = float(np.max(np.abs(merged - single)))
        assert err <= 1e-12, f"partition {part}: merged differs from single pass by {err}"


def check_f16_decoding(orc):
    pattern = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pattern.view(np.float16).astype(np.float64)
    got = np.array([orc.elem_to_double(pattern, i, O.F16) for i in range(65536)])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all(), f"binary16 decoding wrong for {np.count_nonzero(~same)} patterns"


def check_bf16_decoding(orc):
    pattern = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = pattern.view(torch.bfloat16).to(torch.float64).numpy()
    arr = pattern.numpy()
    got = np.array([orc.elem_to_double(arr, i, O.BF16) for i in range(65536)])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all(), f"bfloat16 decoding wrong for {np.count_nonzero(~same)} patterns"


# ---------------------------------------------------------------------------
# worked examples from the pages
# ---------------------------------------------------------------------------
def _write_tokens(orc, pools, slots, tokens_k, tokens_v):
    orc.reshape_and_cache(tokens_k, tokens_v, pools[0], pools[1], np.array(slots, dtype=np.int64))


def check_walkthrough_write(orc, golden):
    ex = golden["block_table_walkthrough"]
    b = ex["block_size"]
    nb = max(ex["free_blocks"]) + 1
    mgr = BlockManager(nb, b, ex["free_blocks"])
    assert mgr.add_sequence(0, ex["prompt_tokens"]) == ex["table_after_prompt"]
    slots = mgr.prompt_slots(0)
    appended = [mgr.append_token(0) for _ in ex["appends"]]
    assert mgr.table(0) == ex["table_after_appends"]
    hkv, d = 2, 8
    total = ex["prompt_tokens"] + len(ex["appends"])
    rng = np.random.default_rng(1)
    tk = rng.standard_normal((total, hkv, d)).astype(np.float32)
    tv = rng.standard_normal((total, hkv, d)).astype(np.float32)
    kp = np.full((nb, hkv, b, d), np.nan, dtype=np.float32)
    vp = kp.copy()
    _write_tokens(orc, (kp, vp), slots + appended, tk, tv)
    for a in ex["appends"]:
        pos = a["position"]
        assert np.array_equal(kp[a["block"], :, a["offset"], :], tk[pos]), \
            f"token {pos} not at block {a['block']} offset {a['offset']}"
        assert np.array_equal(vp[a["block"], :, a["offset"], :], tv[pos])
    # The prompt: block 11 holds tokens 0-3, block 12 holds 4-5 (then 6, 7).
    for pos in range(ex["prompt_tokens"]):
        blk = ex["table_after_prompt"][pos // b]
        assert np.array_equal(kp[blk, :, pos % b, :], tk[pos])
    mgr.free_sequence(0)
    assert sorted(list(mgr.free)[-3:]) == ex["returned_on_finish"]


def check_figure6(orc, golden):
    ex = golden["figure6_decode"]
    b = ex["block_size"]
    mgr = BlockManager(len(ex["free_blocks"]), b, ex["free_blocks"])
    assert mgr.add_sequence(0, ex["prompt_tokens"]) == ex["prompt_table"]
    counts = [sum(1 for p in range(ex["prompt_tokens"]) if p // b == i) for i in range(2)]
    assert counts == ex["tokens_in_prompt_blocks"]
    s1 = mgr.append_token(0)
    s2 = mgr.append_token(0)
    assert mgr.table(0) == ex["table_after"]
    k = np.arange(2 * 4, dtype=np.float32).reshape(2, 1, 4) + 1.0
    kp = np.zeros((len(ex["free_blocks"]), 1, b, 4), dtype=np.float32)
    vp = kp.copy()
    _write_tokens(orc, (kp, vp), [s1, s2], k, -k)
    f, s = ex["first_decode"], ex["second_decode"]
    assert np.array_equal(kp[f["block"], 0, f["offset"]], k[0, 0])
    assert np.array_equal(kp[s["block"], 0, s["offset"]], k[1, 0])
    assert np.array_equal(vp[s["block"], 0, s["offset"]], -k[1, 0])


def check_address_lookup(orc, golden):
    ex = golden["address_lookup"]
    b = ex["block_size"]
    assert blocks_needed(ex["num_tokens"], b) == ex["blocks_needed"]
    for logical, (lo, hi) in enumerate(ex["logical_ranges"]):
        assert all(p // b == logical for p in range(lo, hi + 1))
    # The oracle reads token 5 of a 10-token sequence whose table is 42/07/18
    # from physical block 07: with a single token dominating the scores, the
    # attention output is that block's slot.
    nb = max(ex["table"]) + 1
    d = 4
    kp = np.zeros((nb, 1, b, d), dtype=np.float32)
    vp = np.zeros((nb, 1, b, d), dtype=np.float32)
    off = ex["token_index"] % b
    kp[ex["physical_block"], 0, off, :] = 50.0
    vp[ex["physical_block"], 0, off, :] = [1.0, 2.0, 3.0, 4.0]
    q = np.ones((1, 1, d), dtype=np.float32)
    out = orc.decode(q, kp, vp, O.F32, np.array([ex["table"]], dtype=np.int32),
                     np.array([ex["num_tokens"]], dtype=np.int32), 1, 1.0)
    assert np.max(np.abs(out[0, 0] - [1.0, 2.0, 3.0, 4.0])) < 1e-12


def check_waste_and_sizes(golden):
    ex = golden["internal_waste"]
    b = ex["block_size"]
    c0, c1 = ex["cases"]
    assert blocks_needed(c0["tokens"], b) == c0["blocks"]
    assert c0["tokens"] - c0["full_blocks"] * b == c0["tokens_in_last"]
    assert wasted_slots(c0["tokens"], b) == c0["wasted"]
    assert blocks_needed(c1["tokens"], b) == c1["blocks"]
    assert blocks_needed(c1["tokens"], b) * b == c1["slots"]
    assert ex["requests"] * c1["slots"] == ex["reserved_for_requests"]
    assert max(wasted_slots(n, b) for n in range(1, 200)) == ex["max_waste"]
    kv = golden["kv_size"]
    per_token = metrics.kv_bytes_per_token(kv["num_layers"], 1, kv["hidden_size"], kv["elem_bytes"])
    assert per_token == kv["bytes_per_token"]
    slots = metrics.kv_token_capacity(kv["cache_bytes"], kv["num_layers"], 1, kv["hidden_size"],
                                      kv["elem_bytes"])
    assert round(slots / 1000.0, 1) == kv["slots_thousands"]


def check_copy_on_write(orc, golden):
    ex = golden["copy_on_write"]
    b = ex["block_size"]
    for samples, copies in zip(ex["samples"], ex["copies"]):
        nb = 64
        mgr = BlockManager(nb, b)
        mgr.add_sequence(0, ex["prompt_tokens"])
        for i in range(1, samples):
            mgr.fork(0, i)
        shared_last = mgr.table(0)[-1]
        new_slots = [mgr.append_token(i) for i in range(samples)]
        pairs = mgr.take_copies()
        assert len(pairs) == copies, f"{samples} samples gave {len(pairs)} copies"
        assert all(src == shared_last for src, _ in pairs)
        # the last sample writes in place into the original block
        assert new_slots[-1] // b == shared_last
        # the oracle's copy duplicates K and V of every layer, touching nothing else
        layers, hkv, d = 2, 3, 4
        rng = np.random.default_rng(samples)
        kps = [rng.standard_normal((nb, hkv, b, d)).astype(np.float32) for _ in range(layers)]
        vps = [rng.standard_normal((nb, hkv, b, d)).astype(np.float32) for _ in range(layers)]
        before_k = [p.copy() for p in kps]
        before_v = [p.copy() for p in vps]
        orc.copy_blocks(kps, vps, np.array(pairs, dtype=np.int64))
        dsts = {dst for _, dst in pairs}
        for layer in range(layers):
            for blk in range(nb):
                src = shared_last if blk in dsts else blk
                assert np.array_equal(kps[layer][blk], before_k[layer][src])
                assert np.array_equal(vps[layer][blk], before_v[layer][src])


def check_swap_roundtrip(orc):
    """Swap-out then swap-in restores the blocks; every moved block equals
    numpy's fancy-indexed copy, every other block is untouched."""
    rng = np.random.default_rng(5)
    layers, gpu_nb, host_nb, shape = 2, 12, 7, (3, 4, 8)
    gk = [rng.standard_normal((gpu_nb,) + shape).astype(np.float32) for _ in range(layers)]
    gv = [rng.standard_normal((gpu_nb,) + shape).astype(np.float32) for _ in range(layers)]
    hk = [np.zeros((host_nb,) + shape, np.float32) for _ in range(layers)]
    hv = [np.zeros((host_nb,) + shape, np.float32) for _ in range(layers)]
    out_pairs = np.array([[3, 0], [11, 4], [5, 6]], dtype=np.int64)
    orc.swap_blocks(gk, gv, hk, hv, out_pairs)
    for layer in range(layers):
        assert np.array_equal(hk[layer][out_pairs[:, 1]], gk[layer][out_pairs[:, 0]])
        assert np.array_equal(hv[layer][out_pairs[:, 1]], gv[layer][out_pairs[:, 0]])
        untouched = np.setdiff1d(np.arange(host_nb), out_pairs[:, 1])
        assert not hk[layer][untouched].any()
    # back into different GPU blocks
    back = np.array([[0, 7], [4, 8], [6, 9]], dtype=np.int64)
    gk2 = [x.copy() for x in gk]
    gv2 = [x.copy() for x in gv]
    orc.swap_blocks(hk, hv, gk2, gv2, back)
    for layer in range(layers):
        assert np.array_equal(gk2[layer][[7, 8, 9]], gk[layer][[3, 11, 5]])
        assert np.array_equal(gv2[layer][[7, 8, 9]], gv[layer][[3, 11, 5]])
        keep = [b for b in range(gpu_nb) if b not in (7, 8, 9)]
        assert np.array_equal(gk2[layer][keep], gk[layer][keep])


def _prefill_case(seed, lens, chunks, h, hkv, d, b, code):
    """A paged case whose last chunks[i] tokens of sequence i are its new
    (query) tokens; returns the case and the query rows [sum(chunks)][H][d]."""
    case = paged_case(seed, lens, h, hkv, d, b, code)
    g = torch.Generator().manual_seed(seed + 1)
    q = torch.randn(sum(chunks), h, d, generator=g).to(TORCH_OF[code])
    qs = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    return case, q, qs


def _run_prefill(orc, case, q, qs):
    return orc.prefill(bits(q), qs, bits(case["k_pool"]), bits(case["v_pool"]), case["code"], case["tables"],
                       np.array(case["lens"], dtype=np.int32), case["Hkv"], case["scale"])


def check_prefill_vs_sdpa(orc):
    """Every new token attends to the cached prefix and to the chunk up to
    itself: torch float64 SDPA with that mask, on contiguous K/V."""
    lens, chunks = [40, 7, 64, 33], [17, 7, 1, 32]
    case, q, qs = _prefill_case(701, lens, chunks, 8, 2, 32, 8, O.BF16)
    got = _run_prefill(orc, case, q, qs)
    for i, (n, c) in enumerate(zip(lens, chunks)):
        qi = q[qs[i]:qs[i + 1]].to(torch.float64).permute(1, 0, 2)[None]      # [1, H, c, d]
        k = case["keys"][i].to(torch.float64).permute(1, 0, 2)[None]           # [1, Hkv, n, d]
        v = case["values"][i].to(torch.float64).permute(1, 0, 2)[None]
        pos = torch.arange(n - c, n)[:, None]
        mask = torch.arange(n)[None, :] <= pos                                # [c, n]
        ref = F.scaled_dot_product_attention(qi, k, v, attn_mask=mask, scale=case["scale"], enable_gqa=True)
        err = float(np.max(np.abs(got[qs[i]:qs[i + 1]] - ref[0].permute(1, 0, 2).numpy())))
        assert err <= 1e-12, f"prefill vs SDPA, sequence {i}: {err}"


def check_prefill_special_cases(orc):
    # (a) one new token per sequence is decode
    lens = [5, 40, 17]
    case, q, qs = _prefill_case(702, lens, [1, 1, 1], 4, 2, 16, 8, O.F16)
    got = _run_prefill(orc, case, q, qs)
    dec = orc.decode(bits(q), bits(case["k_pool"]), bits(case["v_pool"]), case["code"], case["tables"],
                     np.array(lens, dtype=np.int32), case["Hkv"], case["scale"])
    assert np.array_equal(got, dec), "a one-token chunk must equal decode"
    # (b) no cached prefix: plain causal self-attention of the chunk
    lens = [23, 9]
    case, q, qs = _prefill_case(703, lens, lens, 4, 4, 16, 4, O.F32)
    got = _run_prefill(orc, case, q, qs)
    for i, n in enumerate(lens):
        qi = q[qs[i]:qs[i + 1]].to(torch.float64).permute(1, 0, 2)[None]
        k = case["keys"][i].to(torch.float64).permute(1, 0, 2)[None]
        v = case["values"][i].to(torch.float64).permute(1, 0, 2)[None]
        ref = F.scaled_dot_product_attention(qi, k, v, is_causal=True, scale=case["scale"])
        assert np.max(np.abs(got[qs[i]:qs[i + 1]] - ref[0].permute(1, 0, 2).numpy())) <= 1e-12


def _numpy_step_pools(w):
    """The pools after the step's copy-on-write copies and cache write, built
    with numpy indexing alone (no oracle code): pairs in list order, then each
    new token's rows at block slot // B, offset slot % B."""
    b = w.block_size
    k, v = bits(w.k_cache).copy(), bits(w.v_cache).copy()
    for src, dst in w.copy_pairs.tolist():
        k[dst] = k[src]
        v[dst] = v[src]
    nk, nv = bits(w.new_key), bits(w.new_value)
    for t, slot in enumerate(w.slot_mapping.tolist()):
        if slot >= 0:
            k[slot // b, :, slot % b, :] = nk[t]
            v[slot // b, :, slot % b, :] = nv[t]
    return k, v


def check_shared_prefix_equals_private_copies(orc):
    """Invariant (3) of paging ("PagedAttention 论文精读笔记", §6.1 and §6.3:
    sequences that share the physical blocks of a common prompt read exactly
    what private copies would hold).  A parallel-sampling step (2 prompts x 8
    samples sharing each 1000-token prompt, copy-on-write of the partial last
    prompt block, per-sample tails) is decoded twice by the oracle: once on
    its own step (its copy, its cache write, the shared tables), once with
    every sequence given private copies of all the blocks it reads, built by
    numpy indexing.  The outputs must be bit-identical."""
    from paged_kv_cache_132_gb300 import workloads

    w = workloads.make("parallel_sampling", device="cpu", num_seqs=16)
    tables = w.block_tables.numpy()
    ctx = w.context_lens.numpy()
    b = w.block_size
    used = [tables[s, : -(-int(ctx[s]) // b)] for s in range(w.num_seqs)]
    counts = np.bincount(np.concatenate(used))
    assert counts.max() >= 8, "the case must share prompt blocks"
    code = code_of(w.dtype)
    # shared: the oracle's whole step
    k, v = bits(w.k_cache).copy(), bits(w.v_cache).copy()
    orc.copy_blocks([k], [v], w.copy_pairs.numpy())
    orc.reshape_and_cache(bits(w.new_key), bits(w.new_value), k, v, w.slot_mapping.numpy())
    shared = orc.decode(bits(w.query), k, v, code, tables, ctx, w.num_kv_heads, w.scale)
    # private: one fresh block per (sequence, logical block)
    kn, vn = _numpy_step_pools(w)
    total = sum(len(u) for u in used)
    kp = np.empty((total,) + kn.shape[1:], dtype=kn.dtype)
    vp = np.empty_like(kp)
    ptab = np.full(tables.shape, -1, dtype=np.int32)
    nxt = 0
    for s, row in enumerate(used):
        for j, blk in enumerate(row):
            kp[nxt], vp[nxt] = kn[blk], vn[blk]
            ptab[s, j] = nxt
            nxt += 1
    private = orc.decode(bits(w.query), kp, vp, code, ptab, ctx, w.num_kv_heads, w.scale)
    assert np.all(np.isfinite(shared)), "a stale (NaN) slot reached a shared-prefix output"
    assert np.array_equal(shared, private), "shared-prefix output differs from private copies"


ORACLE_CHECKS = [check_sdpa, check_weight_sums, check_block_permutation, check_stale_slots_ignored,
                 check_gqa_equals_repeated_mha, check_closed_forms, check_partition_merge,
                 check_f16_decoding, check_bf16_decoding, check_swap_roundtrip,
                 check_prefill_vs_sdpa, check_prefill_special_cases, check_shared_prefix_equals_private_copies]
GOLDEN_CHECKS = [check_walkthrough_write, check_figure6, check_address_lookup, check_copy_on_write]
