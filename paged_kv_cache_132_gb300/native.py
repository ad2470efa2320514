"""ctypes loader of the compiled C-ABI library ``lib/libpa.so`` (see include/pa.h).

There is no fallback: if the library has not been built, every call raises.
Build it with ``python -m paged_kv_cache_132_gb300.build`` (or ``build()`` in
``__graft_entry__``).
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from .build import INCLUDE, LIB_PATH

PA_OK = 0
STATUS_NAMES = {0: "PA_OK", -1: "PA_ERR_INVALID_ARG", -2: "PA_ERR_UNSUPPORTED", -3: "PA_ERR_WORKSPACE",
                -4: "PA_ERR_CUDA", -5: "PA_ERR_DEVICE_FAULT", -6: "PA_ERR_DEVICE_TIMEOUT"}
PA_F32, PA_F16, PA_BF16 = 0, 1, 2
DEVERR_BLOCK_ID, DEVERR_SLOT, DEVERR_CONTEXT_LEN, DEVERR_COPY_PAIR, DEVERR_TIMEOUT = 0x1, 0x2, 0x4, 0x8, 0x10
DEVERR_DUP_SLOT, DEVERR_PAIR_CONFLICT = 0x20, 0x40  # checked mode only
OPT_DEBUG_CHECKS, OPT_DECODE_KERNEL, OPT_DROP_FIRST_FILL = 0, 1, 2  # pa_option
NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024  # PA_NOALLOC_SCRATCH_BYTES


class PaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what} failed: {STATUS_NAMES.get(status, status)}")


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int64), ("num_kv_heads", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def declared_symbols() -> list:
    """Names of the functions include/pa.h declares."""
    with open(os.path.join(INCLUDE, "pa.h"), encoding="utf-8") as f:
        text = f.read()
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(pa_\w+)\s*\(", text, flags=re.M)))


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """The loaded library; raises if it was not built."""
    global _lib
    lib = _lib
    if lib is not None and path == LIB_PATH:
        return lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library not built ({path} missing); run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        desc = ctypes.POINTER(CacheDesc)
        lib.pa_reshape_and_cache.argtypes = [vp, vp, vp, vp, vp, i64, desc, vp]
        lib.pa_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        lib.pa_decode_workspace_size.restype = sz
        lib.pa_decode.argtypes = [vp, i32, vp, vp, vp, desc, vp, i32, vp, i32, i32, i32, i32, ctypes.c_float,
                                  i32, vp, sz, vp]
        lib.pa_decode_noalloc.argtypes = [vp, i32, vp, vp, vp, desc, vp, i32, vp, i32, i32, i32, i32,
                                          ctypes.c_float, i32, vp]
        lib.pa_copy_blocks.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp), i32, vp, i64, desc, vp]
        lib.pa_swap_blocks.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp), i64, ctypes.POINTER(vp),
                                       ctypes.POINTER(vp), i64, i32, vp, i64, desc, vp]
        lib.pa_prefill.argtypes = [vp, i32, vp, vp, i32, i32, vp, vp, desc, vp, i32, vp, i32, i32, i32,
                                   ctypes.c_float, vp]
        lib.pa_get_device_error.argtypes = [vp, ctypes.POINTER(i32)]
        lib.pa_status_string.argtypes = [ctypes.c_int]
        lib.pa_status_string.restype = ctypes.c_char_p
        lib.pa_abi_version.argtypes = []
        lib.pa_set_option.argtypes = [ctypes.c_int, ctypes.c_int]
        lib.pa_get_option.argtypes = [ctypes.c_int]
        for name in ("pa_reshape_and_cache", "pa_decode", "pa_decode_noalloc", "pa_copy_blocks",
                     "pa_swap_blocks", "pa_prefill", "pa_get_device_error", "pa_abi_version", "pa_set_option",
                     "pa_get_option"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib
