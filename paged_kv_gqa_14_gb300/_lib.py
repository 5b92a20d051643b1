"""ctypes loader for the in-tree CUDA library and the raw C-ABI signatures of include/pkv.h.

The library is built by ``paged_kv_gqa_14_gb300.build``.  Loading fails loudly (no CPU
fallback) when it is missing: build it first (``__graft_entry__.build()``).
"""

from __future__ import annotations

import ctypes
import os

from .build import LIB

_c_i64 = ctypes.c_int64
_c_p = ctypes.c_void_p

# name -> (restype, argtypes); mirrors include/pkv.h
SIGNATURES = {
    "pkv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "pkv_version": (ctypes.c_int, []),
    "pkv_kv_append": (
        ctypes.c_int,
        [_c_p, _c_i64, _c_i64, _c_p, _c_i64, _c_i64, _c_p, _c_i64, _c_i64, _c_p, _c_p, _c_p, _c_p,
         _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, ctypes.c_double, _c_p],
    ),
    "pkv_kv_append_paged": (
        ctypes.c_int,
        [_c_p, _c_i64, _c_i64, _c_p, _c_i64, _c_i64, _c_p, _c_i64, _c_i64, _c_p, _c_i64, _c_i64, _c_p, _c_p,
         _c_i64, _c_p, _c_p, _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, ctypes.c_double, _c_p, _c_p, _c_p],
    ),
    "pkv_rope_turn_table": (ctypes.c_int, [ctypes.c_double, _c_i64, ctypes.POINTER(ctypes.c_uint64)]),
    "pkv_paged_attention_workspace_size": (ctypes.c_size_t, [_c_i64] * 6),
    "pkv_paged_attention": (
        ctypes.c_int,
        [_c_p, _c_i64, _c_i64, _c_p, _c_p, _c_i64, _c_i64, _c_p, _c_i64, _c_i64, _c_p, _c_p, _c_i64,
         _c_p, _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, ctypes.c_float, _c_p, ctypes.c_size_t,
         _c_p],
    ),
    "pkv_paged_attention_ex": (
        ctypes.c_int,
        [_c_p, _c_i64, _c_i64, _c_p, _c_p, _c_i64, _c_i64, _c_p, _c_i64, _c_i64, _c_p, _c_p, _c_i64,
         _c_p, _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, ctypes.c_float, _c_p, ctypes.c_size_t,
         _c_p, _c_p],
    ),
    "pkv_paged_attention_workspace_size_ex": (ctypes.c_size_t, [_c_i64] * 6 + [ctypes.c_int32]),
    "pkv_paged_attention_noalloc": (
        ctypes.c_int,
        [_c_p, _c_i64, _c_i64, _c_p, _c_p, _c_i64, _c_i64, _c_p, _c_i64, _c_i64, _c_p, _c_p, _c_i64,
         _c_p, _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, ctypes.c_float, _c_p],
    ),
    "pkv_set_decode_ctas": (ctypes.c_int, [ctypes.c_int32]),
    "pkv_set_fault_injection": (ctypes.c_int, [ctypes.c_int]),
    "pkv_set_overlap": (ctypes.c_int, [ctypes.c_int]),
    "pkv_set_decode_kernel": (ctypes.c_int, [ctypes.c_int]),
    "pkv_set_prefill_kernel": (ctypes.c_int, [ctypes.c_int]),
    "pkv_set_kernel_events": (ctypes.c_int, [ctypes.c_int, _c_p, _c_p]),
    "pkv_get_device_error": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int, _c_p]),
    "pkv_copy": (ctypes.c_int, [_c_p, _c_p, ctypes.c_size_t, _c_p]),
}

STATUS = {
    0: "PKV_OK",
    1: "PKV_ERR_NULL",
    2: "PKV_ERR_SHAPE",
    3: "PKV_ERR_STRIDE",
    4: "PKV_ERR_ALIGN",
    5: "PKV_ERR_UNSUPPORTED",
    6: "PKV_ERR_WORKSPACE",
    7: "PKV_ERR_CUDA",
}

DEVERR = {
    0x1: "PKV_DEVERR_SLOT_RANGE",
    0x2: "PKV_DEVERR_BLOCK_RANGE",
    0x4: "PKV_DEVERR_SPAN",
    0x8: "PKV_DEVERR_CONTEXT",
    0x10: "PKV_DEVERR_TIMEOUT",
}

KERNELS = {"kv_append": 1, "plan": 2, "prefill": 3, "decode": 4}

_lib = None


class AttentionOptions(ctypes.Structure):
    """pkv_attention_options (include/pkv.h)."""

    _fields_ = [("struct_size", ctypes.c_uint32), ("decode_kernel", ctypes.c_int32),
                ("prefill_kernel", ctypes.c_int32), ("overlap", ctypes.c_int32),
                ("decode_ctas", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("side_stream", ctypes.c_void_p), ("fork_event", ctypes.c_void_p),
                ("join_event", ctypes.c_void_p)]


class PkvError(RuntimeError):
    def __init__(self, fn, status, msg):
        super().__init__(f"{fn} failed: {STATUS.get(status, status)} ({msg})")
        self.status = status


def load(path=None):
    """Load (once) and return the ctypes handle of libpkv.so."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB
    if not os.path.exists(p):
        raise RuntimeError(
            f"CUDA library not built: {p} is missing. Build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)."
        )
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    if path is None:
        _lib = lib
    return lib


def check(fn, status):
    if status != 0:
        msg = load().pkv_status_string(status).decode()
        raise PkvError(fn, status, msg)
