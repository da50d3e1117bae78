"""ctypes view of librpa.so (include/rpa.h).  Marshalling only.

The library must be built (``python -m ragged_paged_attention_kv_gb300.build``
or ``__graft_entry__.build()``); loading fails loudly otherwise -- there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "librpa.so")

RPA_OK = 0
RPA_ERR_INVALID_ARG = 1
RPA_ERR_UNSUPPORTED = 2
RPA_ERR_WORKSPACE = 3
RPA_ERR_CUDA = 4
RPA_ERR_NOALLOC_TOO_LARGE = 5

RPA_STATUS_BAD_PAGE = 0x1
RPA_STATUS_BAD_KV_LEN = 0x2
RPA_STATUS_BAD_QUERY_START_LOC = 0x4
RPA_STATUS_BAD_DISTRIBUTION = 0x8
RPA_STATUS_DECODE_QLEN = 0x10
RPA_STATUS_TIMEOUT = 0x20
RPA_STATUS_BAD_SCALE = 0x40

RPA_KV_BF16 = 0
RPA_KV_FP8_E4M3 = 1

# Every symbol include/rpa.h declares.
EXPORTS = ("rpa_workspace_size", "rpa_update_cache", "rpa_forward", "rpa_forward_timed",
           "rpa_forward_noalloc", "rpa_get_status", "rpa_status_string")


class RpaParams(ctypes.Structure):
    """Mirror of rpa_params_t."""
    _fields_ = [
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("pages_per_seq", ctypes.c_int32),
        ("max_num_seqs", ctypes.c_int32),
        ("total_tokens", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32),
        ("sliding_window", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
        ("logits_soft_cap", ctypes.c_float),
        ("k_scale", ctypes.c_float),
        ("v_scale", ctypes.c_float),
        ("k_scale_heads", ctypes.c_void_p),
        ("v_scale_heads", ctypes.c_void_p),
        ("q_scale", ctypes.c_float),
    ]


class RpaError(RuntimeError):
    def __init__(self, func: str, code: int, text: str):
        super().__init__(f"{func} failed: {text} (code {code})")
        self.code = code


_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m ragged_paged_attention_kv_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i32p = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)
        pp = ctypes.POINTER(RpaParams)
        lib.rpa_workspace_size.argtypes = [pp, ctypes.POINTER(ctypes.c_size_t)]
        lib.rpa_workspace_size.restype = ctypes.c_int
        lib.rpa_update_cache.argtypes = [pp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
        lib.rpa_update_cache.restype = ctypes.c_int
        lib.rpa_forward.argtypes = [pp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                    ctypes.c_size_t, vp]
        lib.rpa_forward.restype = ctypes.c_int
        lib.rpa_forward_timed.argtypes = [pp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                          ctypes.c_size_t, vp, ctypes.POINTER(ctypes.c_void_p)]
        lib.rpa_forward_timed.restype = ctypes.c_int
        lib.rpa_forward_noalloc.argtypes = [pp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.rpa_forward_noalloc.restype = ctypes.c_int
        lib.rpa_get_status.argtypes = [vp, vp, i32p]
        lib.rpa_get_status.restype = ctypes.c_int
        lib.rpa_status_string.argtypes = [ctypes.c_int]
        lib.rpa_status_string.restype = ctypes.c_char_p
        _lib = lib
        return lib


def check(func: str, code: int) -> None:
    if code != RPA_OK:
        raise RpaError(func, code, load().rpa_status_string(code).decode())
