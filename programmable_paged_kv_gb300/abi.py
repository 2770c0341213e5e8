"""ctypes declarations of the C ABI in include/pie_fwd.h and include/pie_batcher.h.

Argument marshalling only: every step of the ForwardPass hot path runs in
libpie_fwd.so.  Loading fails loudly when the library has not been built;
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes as C
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpie_fwd.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "pie_fwd.h")
HEADERS = [HEADER, os.path.join(os.path.dirname(HERE), "include", "pie_batcher.h")]

PIE_OK = 0
PIE_EINVAL = -1
PIE_ERANGE = -2
PIE_ENOSPACE = -3
PIE_ECUDA = -4
PIE_EUNSUPPORTED = -5

PIE_F32 = 0
PIE_BF16 = 1

PIE_FOLD_NONE = 0
PIE_FOLD_ALL = 1
PIE_FOLD_COUNT = 2
PIE_FOLD_CHANNEL = 3

PIE_STATUS_FROZEN_WRITE = 1
PIE_STATUS_FOLD_CLAMP = 2
PIE_STATUS_FOLD_GAP = 8
PIE_STATUS_TIMEOUT = 16
PIE_STATUS_NOALLOC_TRUNC = 32
PIE_STATUS_LOOP_FULL = 64


class pie_fwd_desc(C.Structure):
    _fields_ = [("num_q_heads", C.c_int32), ("num_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("page_size", C.c_int32), ("dtype", C.c_int32),
                ("rope_base", C.c_float), ("sm_scale", C.c_float)]


class pie_fwd_meta(C.Structure):
    _fields_ = [("num_lanes", C.c_int32), ("num_rows", C.c_int32),
                ("row_indptr", C.c_void_p), ("positions", C.c_void_p),
                ("slots", C.c_void_p), ("kv_len", C.c_void_p),
                ("page_indptr", C.c_void_p), ("page_ids", C.c_void_p),
                ("num_pool_pages", C.c_int32), ("fold_mode", C.c_void_p),
                ("fold_count", C.c_void_p), ("mask_word_indptr", C.c_void_p),
                ("readout", C.c_void_p), ("num_readout", C.c_int32)]


_P = C.c_void_p
# name -> (restype, argtypes), in header order
SIGNATURES = {
    "pie_fwd_workspace_bytes": (C.c_int, [C.POINTER(pie_fwd_desc), C.POINTER(pie_fwd_meta),
                                          C.POINTER(C.c_size_t)]),
    "pie_fwd_plan": (C.c_int, [C.POINTER(pie_fwd_desc), C.POINTER(pie_fwd_meta), _P, C.c_size_t,
                               _P, C.POINTER(_P)]),
    "pie_fwd_plan_num_readout": (C.c_int32, [_P]),
    "pie_fwd_append_kv": (C.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "pie_fwd_attend": (C.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "pie_fwd_fold": (C.c_int, [_P, _P, _P, _P, _P]),
    "pie_fwd_forward": (C.c_int, [_P, _P, _P, C.c_size_t, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                  _P, _P, _P, _P, _P]),
    "pie_fwd_plan_destroy": (None, [_P]),
    "pie_fwd_last_error": (C.c_char_p, []),
    "pie_fwd_abi_version": (C.c_int, []),
    "pie_fwd_set_timing_events": (C.c_int, [C.c_void_p, C.c_void_p]),
    "pie_fwd_set_mask": (C.c_int, [_P, _P, _P]),
    "pie_fwd_decode_loop_workspace_bytes": (C.c_int, [C.POINTER(pie_fwd_desc), C.c_int32,
                                                      C.c_int32, C.POINTER(C.c_size_t)]),
    "pie_fwd_decode_loop": (C.c_int, [C.POINTER(pie_fwd_desc), C.c_int32, C.c_int32, C.c_void_p,
                                      C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                                      C.c_void_p,
                                      C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                      C.c_void_p, C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p,
                                      C.c_void_p]),
    "pie_fwd_readout_topk_workspace_bytes": (C.c_int, [C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                                                       C.POINTER(C.c_size_t)]),
    "pie_fwd_readout_topk": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_int64,
                                       C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                       C.c_void_p, C.c_size_t, C.c_void_p]),
    "pie_fwd_decode_attend_noalloc": (C.c_int, [C.POINTER(pie_fwd_desc), C.c_int32, C.c_int32,
                                                _P, _P, _P, _P, C.c_int32, _P, _P, _P, _P, _P,
                                                _P, _P]),
    "pie_fwd_test_wait_expiry": (C.c_int, [C.c_int32, C.c_uint32]),
    "pie_fwd_adapter_workspace_bytes": (C.c_int, [C.c_int32, _P, C.c_int32,
                                                  C.POINTER(C.c_size_t)]),
    "pie_fwd_adapter_plan": (C.c_int, [C.c_int32, _P, _P, C.c_int32, C.c_int32, _P, C.c_size_t,
                                       _P, C.POINTER(C.c_void_p)]),
    "pie_fwd_adapter_plan_num_tiles": (C.c_int32, [_P]),
    "pie_fwd_adapter_plan_num_groups": (C.c_int32, [_P]),
    "pie_fwd_adapter_apply": (C.c_int, [_P, C.c_int32, C.c_int32, C.c_int32, C.c_int32, _P, _P,
                                        _P, _P, _P, _P, _P, _P]),
    "pie_fwd_adapter_plan_destroy": (None, [_P]),
    "pie_batcher_create": (C.c_int, [C.c_int32, _P, C.c_int32, C.c_int64, C.POINTER(C.c_void_p)]),
    "pie_batcher_destroy": (None, [_P]),
    "pie_batcher_add_queue": (C.c_int, [_P, C.c_int32, C.POINTER(C.c_int32)]),
    "pie_batcher_submit": (C.c_int, [_P, C.c_int32, C.c_int32, C.c_int64, C.c_int64, _P,
                                     C.c_int32, _P, C.c_int32, _P, C.c_int32,
                                     C.POINTER(C.c_int64)]),
    "pie_batcher_submit_many": (C.c_int, [_P, C.c_int32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                          C.POINTER(C.c_int64)]),
    "pie_batcher_dispatch": (C.c_int, [_P, _P, _P, C.c_int32, C.POINTER(C.c_int32),
                                       C.POINTER(C.c_int32)]),
    "pie_batcher_complete": (C.c_int, [_P, _P, C.c_int32]),
    "pie_batcher_counts": (C.c_int, [_P, C.POINTER(C.c_int64), C.POINTER(C.c_int64)]),
    "pie_batcher_set_pages": (C.c_int, [_P, C.c_int64, _P, C.c_int32]),
    "pie_batcher_submit_forward": (C.c_int, [_P, C.c_int32, _P, C.c_int32, _P, _P, _P, C.c_int32,
                                             C.POINTER(C.c_int64)]),
    "pie_batcher_plan_forward": (C.c_int, [_P, _P, _P, C.c_int32, _P, C.c_int64, _P, C.c_int32,
                                           _P, C.c_size_t, _P, C.POINTER(C.c_void_p), _P, _P, _P,
                                           C.POINTER(C.c_int32), C.POINTER(C.c_int32)]),
    "pie_batcher_forward_pass": (C.c_int, [_P, _P, _P, C.c_int32, _P, C.c_int64, C.c_int32,
                                           C.c_int64, C.c_int64, _P, _P, _P, _P, _P, _P, _P,
                                           C.POINTER(C.c_int32), C.POINTER(C.c_int32),
                                           C.POINTER(C.c_int64)]),
}


def header_functions() -> list:
    """Names of the functions the headers under include/ declare."""
    names = set()
    for h in HEADERS:
        src = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"\b(pie_(?:fwd|batcher)_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


_lib = None


def load(path: str = LIB_PATH):
    """Load libpie_fwd.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library {path} is missing: run "
                           "programmable_paged_kv_gb300.builder.build() first")
    lib = C.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    if path == LIB_PATH:
        _lib = lib
    return lib


class PieError(RuntimeError):
    def __init__(self, code: int, where: str, msg: str):
        super().__init__(f"{where} failed with {code}: {msg}")
        self.code = code


def check(code: int, where: str):
    if code != PIE_OK:
        raise PieError(code, where, load().pie_fwd_last_error().decode())
    return code
