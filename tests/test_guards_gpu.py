"""Guard regions around every buffer a call writes.

No memory checker runs on the GPU machines these tests use, so writes past a
buffer's ends are looked for directly: each pool, output and workspace is a
view into a larger allocation whose margins hold a fixed byte pattern.  After
the call both margins must still hold it, and the results must equal those
of the same call on plain buffers, bit for bit.
"""
import pytest
import torch

from paged_kv_cache_132_gb300 import api, native, workloads

pytestmark = pytest.mark.gpu

MARGIN = 1 << 16       # bytes on each side (a multiple of 256: views keep their alignment)
PATTERN = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _library():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    native.load()


class Guarded:
    """A tensor of `shape`/`dtype` inside a byte buffer with patterned margins."""

    def __init__(self, shape, dtype, device="cuda", pinned=False, init=None):
        n = torch.empty((), dtype=dtype).element_size()
        for s in shape:
            n *= int(s)
        self.nbytes = n
        buf = torch.full((MARGIN + n + MARGIN,), PATTERN, dtype=torch.uint8,
                         device="cpu" if pinned else device)
        self.buf = buf.pin_memory() if pinned else buf
        self.t = self.buf[MARGIN:MARGIN + n].view(dtype).view(tuple(shape))
        if init is not None:
            self.t.copy_(init)

    def intact(self) -> bool:
        lo, hi = self.buf[:MARGIN], self.buf[MARGIN + self.nbytes:]
        return bool((lo == PATTERN).all()) and bool((hi == PATTERN).all())


def same_bits(a: torch.Tensor, b: torch.Tensor) -> bool:
    """Bitwise equality (the pools keep NaN in their unused slots)."""
    return a.shape == b.shape and torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


def _pools(w):
    return (Guarded(w.k_cache.shape, w.k_cache.dtype, init=w.k_cache),
            Guarded(w.v_cache.shape, w.v_cache.dtype, init=w.v_cache))


@pytest.mark.parametrize("name,kw,part,out_dtype", [
    ("tiny", {}, 0, torch.float32),
    ("llama8b", {"num_seqs": 32}, 512, torch.float32),
    ("llama8b", {"num_seqs": 32}, 512, torch.bfloat16),
    ("opt13b", {"num_seqs": 16}, 256, torch.float16),
    ("long_context", {"num_seqs": 4}, 512, torch.float32),
])
def test_write_and_decode_stay_inside(name, kw, part, out_dtype):
    w = workloads.make(name, device="cuda", **kw)
    mc = w.max_context_len
    k, v = _pools(w)
    out = Guarded((w.num_seqs, w.num_heads, w.head_dim), out_dtype)
    ws_bytes = api.decode_workspace_size(w.num_seqs, w.num_heads, mc, part, w.head_dim)
    ws = Guarded((ws_bytes,), torch.uint8)
    api.reshape_and_cache(w.new_key, w.new_value, k.t, v.t, w.slot_mapping)
    api.decode(w.query, k.t, v.t, w.block_tables, w.context_lens, w.scale, out=out.t, out_dtype=out_dtype,
               max_context_len=mc, partition_size=part, workspace=ws.t)
    assert api.get_device_error() == (0, 0)
    assert k.intact() and v.intact(), "pool margins written"
    assert out.intact(), "output margins written"
    assert ws.intact(), "workspace margins written"
    # the same call on plain buffers
    k2, v2 = w.k_cache.clone(), w.v_cache.clone()
    api.reshape_and_cache(w.new_key, w.new_value, k2, v2, w.slot_mapping)
    ref = api.decode(w.query, k2, v2, w.block_tables, w.context_lens, w.scale, out_dtype=out_dtype,
                     max_context_len=mc, partition_size=part)
    assert same_bits(k.t, k2) and same_bits(v.t, v2)
    assert same_bits(out.t, ref)


def test_write_to_first_and_last_slot_stays_inside():
    w = workloads.make("llama8b", device="cuda", num_seqs=4)
    k, v = _pools(w)
    last = w.num_blocks * w.block_size - 1
    slots = torch.tensor([0, last, -1, last - 1], dtype=torch.int64, device="cuda")
    api.reshape_and_cache(w.new_key, w.new_value, k.t, v.t, slots)
    assert api.get_device_error() == (0, 0)
    assert k.intact() and v.intact()
    assert torch.equal(k.t[0, :, 0], w.new_key[0]) and torch.equal(v.t[-1, :, -1], w.new_value[1])


@pytest.mark.parametrize("layers", [1, 3])
def test_copy_blocks_stay_inside(layers):
    w = workloads.make("parallel_sampling", device="cuda")
    ks = [Guarded(w.k_cache.shape, w.k_cache.dtype, init=w.k_cache) for _ in range(layers)]
    vs = [Guarded(w.v_cache.shape, w.v_cache.dtype, init=w.v_cache) for _ in range(layers)]
    api.copy_blocks([g.t for g in ks], [g.t for g in vs], w.copy_pairs)
    assert api.get_device_error() == (0, 0)
    assert all(g.intact() for g in ks + vs)
    k2, v2 = w.k_cache.clone(), w.v_cache.clone()
    api.copy_blocks([k2], [v2], w.copy_pairs)
    assert all(same_bits(g.t, k2) for g in ks) and all(same_bits(g.t, v2) for g in vs)


def test_swap_blocks_stay_inside():
    gen = torch.Generator(device="cuda").manual_seed(5)
    nb, host_nb, shape = 200, 64, (8, 16, 128)
    gk = Guarded((nb,) + shape, torch.bfloat16, init=torch.randn((nb,) + shape, generator=gen, device="cuda"))
    gv = Guarded((nb,) + shape, torch.bfloat16, init=torch.randn((nb,) + shape, generator=gen, device="cuda"))
    hk = Guarded((host_nb,) + shape, torch.bfloat16, pinned=True, init=torch.zeros((host_nb,) + shape))
    hv = Guarded((host_nb,) + shape, torch.bfloat16, pinned=True, init=torch.zeros((host_nb,) + shape))
    # out to the first and last host blocks among others, then back to the GPU pool's ends
    out_pairs = torch.tensor([[3, 0], [nb - 1, host_nb - 1], [100, 30]], dtype=torch.int64, device="cuda")
    api.swap_blocks([gk.t], [gv.t], [hk.t], [hv.t], out_pairs)
    assert api.get_device_error() == (0, 0)
    assert hk.intact() and hv.intact()
    assert torch.equal(hk.t[host_nb - 1], gk.t[nb - 1].cpu()) and torch.equal(hv.t[0], gv.t[3].cpu())
    in_pairs = torch.tensor([[0, 0], [host_nb - 1, nb - 1], [30, 150]], dtype=torch.int64, device="cuda")
    api.swap_blocks([hk.t], [hv.t], [gk.t], [gv.t], in_pairs)
    assert api.get_device_error() == (0, 0)
    assert gk.intact() and gv.intact()
    assert torch.equal(gk.t[0].cpu(), hk.t[0]) and torch.equal(gv.t[150].cpu(), hv.t[30])


@pytest.mark.parametrize("name,kw,out_dtype", [
    ("prefill_tiny", {}, torch.float32),
    ("prefill_llama8b", {"num_seqs": 4}, torch.bfloat16),
    ("prefill_opt13b", {"num_seqs": 3}, torch.float16),
])
def test_prefill_stays_inside(name, kw, out_dtype):
    st = workloads.make_prefill(name, device="cuda", **kw)
    k, v = _pools(st)
    out = Guarded((st.num_tokens, st.num_heads, st.head_dim), out_dtype)
    if st.copy_pairs.numel():
        api.copy_blocks([k.t], [v.t], st.copy_pairs)
    api.reshape_and_cache(st.new_key, st.new_value, k.t, v.t, st.slot_mapping)
    api.prefill(st.query, st.query_start_loc, k.t, v.t, st.block_tables, st.context_lens, st.scale,
                st.max_query_len, out=out.t, out_dtype=out_dtype)
    assert api.get_device_error() == (0, 0)
    assert k.intact() and v.intact() and out.intact()
    k2, v2 = st.k_cache.clone(), st.v_cache.clone()
    if st.copy_pairs.numel():
        api.copy_blocks([k2], [v2], st.copy_pairs)
    api.reshape_and_cache(st.new_key, st.new_value, k2, v2, st.slot_mapping)
    ref = api.prefill(st.query, st.query_start_loc, k2, v2, st.block_tables, st.context_lens, st.scale,
                      st.max_query_len, out_dtype=out_dtype)
    assert same_bits(k.t, k2) and same_bits(v.t, v2)
    assert same_bits(out.t, ref)
