"""Python access to the CPU oracle (``pie_oracle.cpp``).

TEST INFRASTRUCTURE ONLY: the test-suite, the package smoke check and the
benchmark's CPU-baseline leg are the only users.  The CUDA library never
imports this package, and this package never imports the library.

``build()`` compiles the oracle with the host C++ compiler; ``run_pass``
applies one ForwardPass (validate, RoPE + slot scatter, attention, readout,
fold) to numpy pools in place.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pie_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")

OK, EINVAL, ERANGE = 0, -1, -2
ST_FROZEN_WRITE, ST_FOLD_CLAMP, ST_FOLD_GAP = 1, 2, 8


class _Desc(C.Structure):
    _fields_ = [("num_q_heads", C.c_int32), ("num_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("page_size", C.c_int32), ("dtype", C.c_int32),
                ("rope_base", C.c_double), ("sm_scale", C.c_double)]


class _Meta(C.Structure):
    _fields_ = [("num_lanes", C.c_int32), ("num_rows", C.c_int32),
                ("row_indptr", C.c_void_p), ("positions", C.c_void_p),
                ("slots", C.c_void_p), ("kv_len", C.c_void_p),
                ("page_indptr", C.c_void_p), ("page_ids", C.c_void_p),
                ("num_pool_pages", C.c_int32), ("fold_mode", C.c_void_p),
                ("fold_count", C.c_void_p), ("mask_word_indptr", C.c_void_p),
                ("readout", C.c_void_p), ("num_readout", C.c_int32)]


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source (plain -O2, no vector ISA flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-o", tmp,
                               _SRC, "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def load(path: str):
    """Load an oracle shared library from `path` and declare its signatures."""
    L = C.CDLL(path)
    _declare(L)
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = load(build())
    return _lib


def _declare(L):
    L.orc_validate.restype = C.c_int
    L.orc_validate.argtypes = [C.POINTER(_Desc), C.POINTER(_Meta)]
    L.orc_append_kv.restype = None
    L.orc_append_kv.argtypes = [C.POINTER(_Desc), C.POINTER(_Meta)] + [C.c_void_p] * 8
    L.orc_attend.restype = None
    L.orc_attend.argtypes = ([C.POINTER(_Desc), C.POINTER(_Meta)] + [C.c_void_p] * 5 +
                             [C.c_int32, C.c_void_p, C.c_void_p, C.c_int32])
    L.orc_readout_rows.restype = C.c_int32
    L.orc_readout_rows.argtypes = [C.POINTER(_Meta), C.c_void_p, C.c_int32]
    L.orc_fold.restype = None
    L.orc_fold.argtypes = [C.POINTER(_Meta), C.c_void_p, C.c_void_p, C.c_void_p]
    L.orc_kv_bytes.restype = C.c_int64
    L.orc_kv_bytes.argtypes = [C.c_int64] * 5
    L.orc_page_waste.restype = C.c_int64
    L.orc_page_waste.argtypes = [C.c_int64] * 2
    L.orc_round_bf16.restype = C.c_uint16
    L.orc_round_bf16.argtypes = [C.c_double]
    L.orc_rope.restype = None
    L.orc_rope.argtypes = [C.POINTER(_Desc), C.c_void_p, C.c_int32, C.c_void_p]


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def make_desc(desc) -> _Desc:
    return _Desc(desc.num_q_heads, desc.num_kv_heads, desc.head_dim, desc.page_size,
                 desc.dtype, float(desc.rope_base), float(desc.sm_scale))


class Meta:
    """Keeps the numpy arrays alive while ctypes holds their addresses."""

    def __init__(self, p, page_ids=None, num_pool_pages=0, use_mask=True):
        self.arrs = dict(
            row_indptr=np.ascontiguousarray(p.row_indptr, np.int32),
            positions=np.ascontiguousarray(p.positions, np.int32),
            slots=np.ascontiguousarray(p.slots, np.int32),
            kv_len=np.ascontiguousarray(p.kv_len, np.int32),
            page_indptr=np.ascontiguousarray(p.page_indptr, np.int32),
            page_ids=np.ascontiguousarray(p.page_ids if page_ids is None else page_ids, np.int32),
            fold_mode=np.ascontiguousarray(p.fold_mode, np.int32),
            fold_count=np.ascontiguousarray(p.fold_count, np.int32),
        )
        mwi = p.mask_word_indptr if use_mask else None
        self.arrs["mask_word_indptr"] = None if mwi is None else np.ascontiguousarray(mwi, np.int64)
        ro = p.readout
        self.arrs["readout"] = None if ro is None else np.ascontiguousarray(ro, np.int32)
        a = self.arrs
        self.c = _Meta(int(p.kv_len.shape[0]), int(p.positions.shape[0]),
                       _ptr(a["row_indptr"]), _ptr(a["positions"]), _ptr(a["slots"]),
                       _ptr(a["kv_len"]), _ptr(a["page_indptr"]), _ptr(a["page_ids"]),
                       int(num_pool_pages), _ptr(a["fold_mode"]), _ptr(a["fold_count"]),
                       _ptr(a["mask_word_indptr"]), _ptr(a["readout"]),
                       0 if ro is None else int(ro.shape[0]))


def validate(desc, p, page_ids=None, num_pool_pages=None) -> int:
    npp = num_pool_pages if num_pool_pages is not None else int(np.max(p.page_ids, initial=-1)) + 1
    m = Meta(p, page_ids, npp)
    return lib().orc_validate(C.byref(make_desc(desc)), C.byref(m.c))


def kv_bytes(layers, kv_heads, head_dim, tokens, elem_bytes) -> int:
    return int(lib().orc_kv_bytes(layers, kv_heads, head_dim, tokens, elem_bytes))


def page_waste(tokens, page_size) -> int:
    return int(lib().orc_page_waste(tokens, page_size))


def round_bf16(x: float) -> int:
    return int(lib().orc_round_bf16(float(x)))


def rope(desc, x: np.ndarray, pos: int) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float64)
    out = np.zeros_like(x)
    lib().orc_rope(C.byref(make_desc(desc)), x.ctypes.data, int(pos), out.ctypes.data)
    return out


def run_pass(desc, p, k_pool: np.ndarray, v_pool: np.ndarray, frozen_len: np.ndarray,
             page_ids: Optional[np.ndarray] = None, rows: Optional[np.ndarray] = None,
             channel: Optional[np.ndarray] = None, num_threads: int = 1,
             use_mask: bool = True, do_fold: bool = True) -> dict:
    """Apply one pass to the (compact) pools in place.

    page_ids: page ids indexing k_pool/v_pool (defaults to p.page_ids).
    rows: rows whose attention is computed (default all); other rows' outputs
          are left as NaN.
    Returns q_rot (storage dtype), out [N,Hq,d] and lse [N,Hq] (float64),
    readout row indices, status bits and the error code of validation.
    """
    L = lib()
    d = make_desc(desc)
    m = Meta(p, page_ids, k_pool.shape[0], use_mask)
    res = {"err": L.orc_validate(C.byref(d), C.byref(m.c))}
    if res["err"] != OK:
        return res
    N, Hq, D = p.num_rows, desc.num_q_heads, desc.head_dim
    status = np.zeros(1, np.uint32)
    q_rot = np.zeros_like(p.q)
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    assert frozen_len.dtype == np.int32 and frozen_len.flags.c_contiguous
    L.orc_append_kv(C.byref(d), C.byref(m.c), _ptr(np.ascontiguousarray(p.q)),
                    _ptr(np.ascontiguousarray(p.k)), _ptr(np.ascontiguousarray(p.v)),
                    _ptr(q_rot), _ptr(k_pool), _ptr(v_pool), _ptr(frozen_len), _ptr(status))
    out = np.full((N, Hq, D), np.nan, np.float64)
    lse = np.full((N, Hq), np.nan, np.float64)
    mw = None
    if use_mask and p.mask_words is not None:
        mw = np.ascontiguousarray(p.mask_words, np.uint32)
    sel = None if rows is None else np.ascontiguousarray(rows, np.int32)
    L.orc_attend(C.byref(d), C.byref(m.c), _ptr(q_rot), _ptr(k_pool), _ptr(v_pool), _ptr(mw),
                 _ptr(sel), 0 if sel is None else int(sel.shape[0]), _ptr(out), _ptr(lse),
                 int(num_threads))
    cap = max(1, N + p.num_lanes)
    ro = np.zeros(cap, np.int32)
    R = L.orc_readout_rows(C.byref(m.c), _ptr(ro), cap)
    if do_fold:
        ch = channel if channel is not None else p.channel
        ch = None if ch is None else np.ascontiguousarray(ch, np.int32)
        L.orc_fold(C.byref(m.c), _ptr(frozen_len), _ptr(ch), _ptr(status))
    res.update(q_rot=q_rot, out=out, lse=lse, readout_rows=ro[:R].copy(),
               status=int(status[0]))
    return res


def run_scenario(sc, num_threads: int = 1, rows_per_pass=None, use_mask: bool = True):
    """Run every pass of a workloads.Scenario on compact copies of its pool.

    Returns (k_pool, v_pool, frozen_len, [per-pass results])."""
    k_pool = sc.k_init.copy()
    v_pool = sc.v_init.copy()
    frozen = sc.frozen_len0.copy()
    results = []
    for i, p in enumerate(sc.passes):
        rows = None if rows_per_pass is None else rows_per_pass[i]
        r = run_pass(sc.desc, p, k_pool, v_pool, frozen, page_ids=sc.compact_page_ids(p.page_ids),
                     rows=rows, num_threads=num_threads, use_mask=use_mask)
        assert r["err"] == OK, (sc.name, i, r["err"])
        results.append(r)
    return k_pool, v_pool, frozen, results
