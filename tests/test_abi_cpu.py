"""The C-ABI library without a GPU: it loads, exports every declared symbol,
and rejects bad arguments on the host before any CUDA call (CPU only)."""
import ctypes
import os
import subprocess
import sys

import pytest

from paged_kv_cache_132_gb300 import build, native


@pytest.fixture(scope="module")
def lib():
    build.build_library()
    return native.load()


def test_exports_every_declared_symbol(lib):
    names = native.declared_symbols()
    assert set(names) >= {"pa_reshape_and_cache", "pa_decode", "pa_copy_blocks", "pa_decode_workspace_size",
                          "pa_get_device_error", "pa_status_string", "pa_abi_version"}
    for name in names:
        assert hasattr(lib, name), f"{name} declared in include/pa.h but not exported"


def test_version_and_status_strings(lib):
    assert lib.pa_abi_version() == 2
    for code, name in native.STATUS_NAMES.items():
        assert lib.pa_status_string(code).decode() == name
    assert lib.pa_status_string(-99).decode() == "PA_ERR_UNKNOWN"


def test_workspace_size(lib):
    ws = lib.pa_decode_workspace_size
    assert ws(4, 4, 64, 0, 64) > 0
    # grows with the number of partitions
    assert ws(16, 32, 32768, 512, 128) > ws(16, 32, 512, 512, 128)
    # at least the partial outputs: S * H * parts * d floats
    assert ws(16, 32, 32768, 512, 128) >= 16 * 32 * 64 * 128 * 4
    # invalid arguments -> 0
    assert ws(-1, 4, 64, 0, 64) == 0
    assert ws(4, 0, 64, 0, 64) == 0
    assert ws(4, 4, 64, 100, 64) == 0   # partition not a multiple of 64
    assert ws(4, 4, -5, 0, 64) == 0


FAKE = 0x10000  # aligned, never dereferenced: every case below fails validation first


def _desc(nb=8, hkv=2, bs=16, d=64, dtype=native.PA_BF16):
    return native.CacheDesc(nb, hkv, bs, d, dtype)


def _decode(lib, **over):
    a = dict(out=FAKE, out_dtype=native.PA_F32, query=FAKE, k=FAKE, v=FAKE, desc=_desc(), tables=FAKE,
             max_blocks=4, ctx=FAKE, num_seqs=2, max_ctx=64, num_heads=4, num_kv_heads=2, scale=0.125,
             part=0, ws=FAKE, ws_bytes=0, stream=None)
    a.update(over)
    return lib.pa_decode(a["out"], a["out_dtype"], a["query"], a["k"], a["v"], ctypes.byref(a["desc"]),
                         a["tables"], a["max_blocks"], a["ctx"], a["num_seqs"], a["max_ctx"], a["num_heads"],
                         a["num_kv_heads"], a["scale"], a["part"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("over,status", [
    (dict(desc=_desc(nb=0)), -1),
    (dict(desc=_desc(dtype=7)), -1),
    (dict(desc=_desc(d=60)), -1),              # 120 bytes: not a multiple of 16
    (dict(out_dtype=5), -1),
    (dict(num_kv_heads=3), -1),                # differs from the pool
    (dict(num_heads=5), -1),                   # not a multiple of num_kv_heads
    (dict(query=FAKE + 8), -1),                # misaligned
    (dict(out=0), -1),
    (dict(tables=FAKE + 2), -1),
    (dict(part=96), -1),
    (dict(scale=float("nan")), -1),
    (dict(max_blocks=0), -1),
    (dict(num_heads=32, num_kv_heads=2), -2),  # group 16
    (dict(desc=_desc(d=96)), -2),
    (dict(desc=_desc(bs=64)), -2),
    (dict(desc=_desc(bs=4)), -2),
])
def test_decode_rejects_on_host(lib, over, status):
    assert _decode(lib, **over) == status


def test_decode_empty_batch_is_noop(lib):
    assert _decode(lib, num_seqs=0) == 0


def test_reshape_and_cache_rejects_on_host(lib):
    d = _desc()
    f = lib.pa_reshape_and_cache
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, -1, ctypes.byref(d), None) == -1
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 0, ctypes.byref(d), None) == 0     # no tokens: no-op
    assert f(FAKE + 4, FAKE, FAKE, FAKE, FAKE, 3, ctypes.byref(d), None) == -1
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE + 4, 3, ctypes.byref(d), None) == -1
    bad = _desc(hkv=0)
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 3, ctypes.byref(bad), None) == -1


def test_copy_blocks_rejects_on_host(lib):
    d = _desc()
    ptrs = (ctypes.c_void_p * 2)(FAKE, FAKE)
    f = lib.pa_copy_blocks
    assert f(ptrs, ptrs, 0, FAKE, 3, ctypes.byref(d), None) == -1      # no layers
    assert f(ptrs, ptrs, 257, FAKE, 3, ctypes.byref(d), None) == -1    # too many layers
    assert f(ptrs, ptrs, 2, FAKE, -1, ctypes.byref(d), None) == -1
    assert f(ptrs, ptrs, 2, FAKE, 0, ctypes.byref(d), None) == 0       # nothing to copy
    assert f(ptrs, ptrs, 2, FAKE + 4, 3, ctypes.byref(d), None) == -1
    mis = (ctypes.c_void_p * 2)(FAKE, FAKE + 8)
    assert f(mis, ptrs, 2, FAKE, 3, ctypes.byref(d), None) == -1


def test_get_device_error_needs_output(lib):
    assert lib.pa_get_device_error(None, None) == -1


def test_swap_blocks_rejects_on_host(lib):
    d = _desc()
    ptrs = (ctypes.c_void_p * 2)(FAKE, FAKE)
    f = lib.pa_swap_blocks
    assert f(ptrs, ptrs, 8, ptrs, ptrs, 8, 0, FAKE, 3, ctypes.byref(d), None) == -1      # no layers
    assert f(ptrs, ptrs, 0, ptrs, ptrs, 8, 2, FAKE, 3, ctypes.byref(d), None) == -1      # empty source pool
    assert f(ptrs, ptrs, 8, ptrs, ptrs, 8, 2, FAKE, 0, ctypes.byref(d), None) == 0       # nothing to move
    assert f(ptrs, ptrs, 8, ptrs, ptrs, 8, 2, FAKE + 4, 3, ctypes.byref(d), None) == -1  # misaligned pairs
    mis = (ctypes.c_void_p * 2)(FAKE, FAKE + 8)
    assert f(ptrs, ptrs, 8, mis, ptrs, 8, 2, FAKE, 3, ctypes.byref(d), None) == -1


def _prefill(lib, **over):
    a = dict(out=FAKE, out_dtype=native.PA_F32, query=FAKE, qsl=FAKE, tokens=40, max_q=20, k=FAKE, v=FAKE,
             desc=_desc(), tables=FAKE, max_blocks=4, ctx=FAKE, num_seqs=2, num_heads=4, num_kv_heads=2,
             scale=0.125, stream=None)
    a.update(over)
    return lib.pa_prefill(a["out"], a["out_dtype"], a["query"], a["qsl"], a["tokens"], a["max_q"], a["k"], a["v"],
                          ctypes.byref(a["desc"]), a["tables"], a["max_blocks"], a["ctx"], a["num_seqs"],
                          a["num_heads"], a["num_kv_heads"], a["scale"], a["stream"])


@pytest.mark.parametrize("over,status", [
    (dict(desc=_desc(nb=0)), -1),
    (dict(out_dtype=9), -1),
    (dict(num_kv_heads=3), -1),
    (dict(num_heads=5), -1),                    # not a multiple of num_kv_heads
    (dict(tokens=-1), -1),
    (dict(max_q=-2), -1),
    (dict(max_blocks=0), -1),
    (dict(scale=float("inf")), -1),
    (dict(scale=0.0), -1),
    (dict(scale=-0.125), -1),
    (dict(query=FAKE + 8), -1),                 # misaligned
    (dict(qsl=FAKE + 2), -1),
    (dict(out=0), -1),
    (dict(desc=_desc(dtype=native.PA_F32)), -2),  # tensor cores: 16-bit pools only
    (dict(num_heads=32, num_kv_heads=2), -2),   # group 16
    (dict(desc=_desc(d=96)), -2),
    (dict(desc=_desc(bs=4)), -2),
])
def test_prefill_rejects_on_host(lib, over, status):
    assert _prefill(lib, **over) == status


def test_prefill_nothing_to_do_is_noop(lib):
    assert _prefill(lib, num_seqs=0) == 0
    assert _prefill(lib, tokens=0) == 0
    assert _prefill(lib, max_q=0) == 0


def test_options_set_get_and_restore(lib):
    for opt in (native.OPT_DEBUG_CHECKS, native.OPT_DECODE_KERNEL, native.OPT_DROP_FIRST_FILL):
        before = lib.pa_get_option(opt)
        assert before in (0, 1)
        assert lib.pa_set_option(opt, 1) == before
        assert lib.pa_get_option(opt) == 1
        assert lib.pa_set_option(opt, 0) == 1
        assert lib.pa_get_option(opt) == 0
        lib.pa_set_option(opt, before)
    assert lib.pa_set_option(3, 1) == -1      # unknown option
    assert lib.pa_set_option(-1, 0) == -1
    assert lib.pa_set_option(0, 2) == -1      # options are 0 or 1
    assert lib.pa_get_option(7) == -1


def test_option_api_context_manager(lib):
    from paged_kv_cache_132_gb300 import api

    assert not api.get_option("debug_checks")
    with api.option("debug_checks"):
        assert api.get_option("debug_checks")
        with api.option("debug_checks", False):
            assert not api.get_option("debug_checks")
        assert api.get_option("debug_checks")
    assert not api.get_option("debug_checks")


_ENV_SCRIPT = """
import sys
sys.path.insert(0, {root!r})
from paged_kv_cache_132_gb300 import native
lib = native.load()
print(lib.pa_get_option(native.OPT_DEBUG_CHECKS), lib.pa_get_option(native.OPT_DECODE_KERNEL),
      lib.pa_get_option(native.OPT_DROP_FIRST_FILL))
lib.pa_set_option(native.OPT_DEBUG_CHECKS, 0)
print(lib.pa_get_option(native.OPT_DEBUG_CHECKS))
"""


@pytest.mark.parametrize("env,expect", [
    ({"PA_DEBUG_CHECKS": "1", "PA_DECODE_KERNEL": "simt", "PA_DEBUG_DROP_FIRST_FILL": "1"}, "1 1 1"),
    ({"PA_DEBUG_CHECKS": "0", "PA_DECODE_KERNEL": "mma"}, "0 0 0"),
    ({}, "0 0 0"),
])
def test_options_start_from_the_environment(lib, env, expect):
    """Each option's first value comes from its environment variable, read
    once; pa_set_option overrides it afterwards."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    full = {k: v for k, v in os.environ.items()
            if k not in ("PA_DEBUG_CHECKS", "PA_DECODE_KERNEL", "PA_DEBUG_DROP_FIRST_FILL")}
    full.update(env)
    r = subprocess.run([sys.executable, "-c", _ENV_SCRIPT.format(root=root)], env=full, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    lines = r.stdout.split("\n")
    assert lines[0].strip() == expect
    assert lines[1].strip() == "0"
