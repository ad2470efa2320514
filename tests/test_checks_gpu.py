"""Checked mode (PA_OPT_DEBUG_CHECKS) on the GPU.

The cache write and the copy-on-write copies run their entries in parallel,
which is exact only when slots are distinct and copies independent (distinct
destinations, no destination that any copy reads; "PagedAttention 论文精读笔记",
§6.1).  With the option on, each call first runs a pre-pass that reports a
broken precondition through the device error word, never by trapping.  Each
test feeds one violation, reads the expected bit, then runs a clean call on the
same context and reads no error.
"""
import pytest
import torch

from paged_kv_cache_132_gb300 import api, native, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    native.load()


@pytest.fixture
def checked():
    api.get_device_error()  # start from a clean error word
    with api.option("debug_checks"):
        yield
    assert api.get_device_error() == (0, 0)


def _tiny():
    w = workloads.make("tiny", device="cuda")
    return w, w.k_cache.clone(), w.v_cache.clone()


def _clean_step(w, k, v):
    """A valid step on the same context: no error bit may appear."""
    api.reshape_and_cache(w.new_key, w.new_value, k, v, w.slot_mapping)
    out = api.decode(w.query, k, v, w.block_tables, w.context_lens, w.scale, max_context_len=w.max_context_len)
    assert api.get_device_error() == (0, 0)
    assert torch.isfinite(out).all()


def test_duplicate_slot_is_reported(checked):
    w, k, v = _tiny()
    slots = w.slot_mapping.clone()
    slots[2] = slots[0]
    api.reshape_and_cache(w.new_key, w.new_value, k, v, slots)
    status, code = api.get_device_error()
    assert status == -5 and code == native.DEVERR_DUP_SLOT
    _clean_step(w, w.k_cache.clone(), w.v_cache.clone())


def test_negative_slots_may_repeat(checked):
    w, k, v = _tiny()
    slots = w.slot_mapping.clone()
    slots[1] = -1
    slots[3] = -1
    api.reshape_and_cache(w.new_key, w.new_value, k, v, slots)
    assert api.get_device_error() == (0, 0)


def test_distinct_slots_of_a_prefill_batch_pass(checked):
    st = workloads.make_prefill("prefill_llama8b", device="cuda", num_seqs=8)
    k, v = st.k_cache.clone(), st.v_cache.clone()
    assert st.slot_mapping.numel() > 2000
    api.copy_blocks([k], [v], st.copy_pairs)
    api.reshape_and_cache(st.new_key, st.new_value, k, v, st.slot_mapping)
    assert api.get_device_error() == (0, 0)
    # the same batch with its last token's slot repeated at the front
    slots = st.slot_mapping.clone()
    slots[0] = slots[-1]
    api.reshape_and_cache(st.new_key, st.new_value, k, v, slots)
    status, code = api.get_device_error()
    assert status == -5 and code == native.DEVERR_DUP_SLOT


@pytest.mark.parametrize("pairs", [
    [[0, 5], [1, 5]],          # destination repeated
    [[3, 3]],                  # a block onto itself
    [[0, 5], [5, 6]],          # a destination that another pair reads
    [[7, 8], [2, 9], [9, 1]],  # the same, later in the list
])
def test_conflicting_copy_pairs_are_reported(checked, pairs):
    w, k, v = _tiny()
    p = torch.tensor(pairs, dtype=torch.int64, device="cuda")
    api.copy_blocks([k], [v], p)
    status, code = api.get_device_error()
    assert status == -5 and code == native.DEVERR_PAIR_CONFLICT
    _clean_step(w, w.k_cache.clone(), w.v_cache.clone())


def test_independent_copy_pairs_pass(checked):
    w = workloads.make("parallel_sampling", device="cuda")
    k, v = w.k_cache.clone(), w.v_cache.clone()
    assert w.copy_pairs.shape[0] == 224  # one source, many destinations: allowed
    api.copy_blocks([k], [v], w.copy_pairs)
    assert api.get_device_error() == (0, 0)


def test_swap_pairs(checked):
    w, k, v = _tiny()
    hk = torch.zeros((4,) + tuple(k.shape[1:]), dtype=k.dtype).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    # between two pools a destination may equal a source id
    ok = torch.tensor([[0, 1], [1, 0], [3, 2]], dtype=torch.int64, device="cuda")
    api.swap_blocks([k], [v], [hk], [hv], ok)
    assert api.get_device_error() == (0, 0)
    dup = torch.tensor([[0, 1], [2, 1]], dtype=torch.int64, device="cuda")
    api.swap_blocks([k], [v], [hk], [hv], dup)
    status, code = api.get_device_error()
    assert status == -5 and code == native.DEVERR_PAIR_CONFLICT
    # within one pool the copy rules apply
    same = torch.tensor([[4, 6], [6, 7]], dtype=torch.int64, device="cuda")
    api.swap_blocks([k], [v], [k], [v], same)
    status, code = api.get_device_error()
    assert status == -5 and code == native.DEVERR_PAIR_CONFLICT


def test_context_above_max_context_len_is_reported(checked):
    # Lengths within the table's capacity and the workspace, but above the
    # bound the call was sized with: only the checked mode sees it.
    w = workloads.make("llama8b", device="cuda", num_seqs=8)
    k, v = w.k_cache.clone(), w.v_cache.clone()
    api.reshape_and_cache(w.new_key, w.new_value, k, v, w.slot_mapping)
    mc = int(w.context_lens.max())
    api.decode(w.query, k, v, w.block_tables, w.context_lens, w.scale, max_context_len=mc - 1,
               partition_size=4096 * 16)
    status, code = api.get_device_error()
    assert status == -5 and code == native.DEVERR_CONTEXT_LEN
    api.decode(w.query, k, v, w.block_tables, w.context_lens, w.scale, max_context_len=mc)
    assert api.get_device_error() == (0, 0)


def test_bad_block_id_is_reported_by_the_check(checked):
    w, k, v = _tiny()
    tables = w.block_tables.clone()
    tables[3, 0] = -2
    api.decode(w.query, k, v, tables, w.context_lens, w.scale, max_context_len=64)
    status, code = api.get_device_error()
    assert status == -5 and code & native.DEVERR_BLOCK_ID


def test_checks_off_by_default():
    """Without the option, a repeated slot is not looked for (the default
    path launches no pre-pass)."""
    assert not api.get_option("debug_checks")
    w, k, v = _tiny()
    slots = w.slot_mapping.clone()
    slots[2] = slots[0]
    api.reshape_and_cache(w.new_key, w.new_value, k, v, slots)
    assert api.get_device_error() == (0, 0)


def test_checked_step_matches_unchecked():
    """The pre-passes change nothing in the results."""
    w = workloads.make("llama8b", device="cuda", num_seqs=32)
    outs = []
    for on in (False, True):
        k, v = w.k_cache.clone(), w.v_cache.clone()
        with api.option("debug_checks", on):
            api.reshape_and_cache(w.new_key, w.new_value, k, v, w.slot_mapping)
            outs.append(api.decode(w.query, k, v, w.block_tables, w.context_lens, w.scale,
                                   max_context_len=w.max_context_len, partition_size=512))
            assert api.get_device_error() == (0, 0)
    assert torch.equal(outs[0], outs[1])


def _pair_conflict(pairs, same_pool=True):
    """Whether a pair list breaks the copy preconditions (plain Python)."""
    dsts = [d for _, d in pairs]
    if len(set(dsts)) != len(dsts):
        return True
    return same_pool and bool(set(dsts) & {s for s, _ in pairs})


@pytest.mark.parametrize("seed", range(12))
def test_random_lists_flag_exactly_the_violations(checked, seed):
    """Random slot and pair lists, about half of them valid: the checked mode
    sets its bit exactly when the list breaks a precondition."""
    g = torch.Generator().manual_seed(seed)
    w, k, v = _tiny()
    nslots = w.num_blocks * w.block_size
    n = int(torch.randint(1, 300, (1,), generator=g))
    slots = torch.randperm(nslots * 8, generator=g)[:n] % nslots if seed % 2 else torch.randperm(nslots, generator=g)[:min(n, nslots)]
    slots = slots.to(torch.int64)
    slots[torch.rand(slots.numel(), generator=g) < 0.1] = -1  # padding tokens never conflict
    valid = slots[slots >= 0]
    expect = bool(valid.unique().numel() != valid.numel())
    keys = torch.randn(slots.numel(), 4, 64, generator=g).cuda()
    api.reshape_and_cache(keys, keys, k, v, slots.cuda())
    status, code = api.get_device_error()
    assert (code == native.DEVERR_DUP_SLOT) == expect and (status == -5) == expect, (seed, expect, code)
    m = int(torch.randint(1, 40, (1,), generator=g))
    pairs = torch.randint(0, w.num_blocks, (m, 2), generator=g)
    if seed % 3 == 0:  # a valid list: distinct destinations, disjoint from the sources
        blocks = torch.randperm(w.num_blocks, generator=g)
        m = min(m, w.num_blocks // 2)
        pairs = torch.stack([blocks[:m], blocks[m:2 * m]], dim=1)
    expect = _pair_conflict(pairs.tolist())
    api.copy_blocks([k], [v], pairs.cuda())
    status, code = api.get_device_error()
    assert (code == native.DEVERR_PAIR_CONFLICT) == expect and (status == -5) == expect, (seed, expect, code)
