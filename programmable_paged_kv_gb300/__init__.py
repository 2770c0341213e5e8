"""GB300 (sm_103a) ForwardPass hot path: RoPE + slot scatter, paged GQA
attention under per-row slot masks, readout and fold, behind a C ABI
(include/pie_fwd.h).

This package is a thin binding: it marshals host metadata (numpy arrays)
and torch device tensors into the C entry points of libpie_fwd.so.  PyTorch
only provides device memory and the current stream.  There is no fallback:
if the library is missing every call raises.
"""
from __future__ import annotations

import ctypes as C
import types
from typing import Optional

import numpy as np

from . import abi
from .abi import (PIE_BF16, PIE_F32, PIE_FOLD_ALL, PIE_FOLD_CHANNEL, PIE_FOLD_COUNT,
                  PIE_FOLD_NONE, PIE_STATUS_FOLD_CLAMP, PIE_STATUS_FOLD_GAP,
                  PIE_STATUS_FROZEN_WRITE, PIE_STATUS_TIMEOUT, PieError)

__all__ = ["ForwardPlan", "PieError", "make_desc", "make_meta", "workspace_bytes", "build",
           "set_timing_events", "readout_topk", "readout_topk_workspace_bytes",
           "decode_loop", "decode_loop_workspace_bytes", "AdapterPlan", "adapter_workspace_bytes",
           "Batcher",
           "PIE_F32", "PIE_BF16", "PIE_FOLD_NONE", "PIE_FOLD_ALL", "PIE_FOLD_COUNT",
           "PIE_FOLD_CHANNEL", "PIE_STATUS_FROZEN_WRITE", "PIE_STATUS_FOLD_CLAMP",
           "PIE_STATUS_FOLD_GAP", "PIE_STATUS_TIMEOUT"]


def build(force: bool = False) -> str:
    from .builder import build as _b
    return _b(force=force)


def make_desc(d) -> abi.pie_fwd_desc:
    """From any object with num_q_heads, num_kv_heads, head_dim, page_size,
    dtype (PIE_F32 / PIE_BF16), rope_base and sm_scale attributes."""
    return abi.pie_fwd_desc(int(d.num_q_heads), int(d.num_kv_heads), int(d.head_dim),
                            int(d.page_size), int(d.dtype), float(d.rope_base),
                            float(getattr(d, "sm_scale", 0.0)))


class _HostMeta:
    """pie_fwd_meta over numpy arrays that stay alive with this object."""

    def __init__(self, row_indptr, positions, slots, kv_len, page_indptr, page_ids,
                 num_pool_pages, fold_mode, fold_count=None, mask_word_indptr=None,
                 readout=None):
        i32 = lambda a: None if a is None else np.ascontiguousarray(a, dtype=np.int32)
        self.keep = dict(row_indptr=i32(row_indptr), positions=i32(positions), slots=i32(slots),
                         kv_len=i32(kv_len), page_indptr=i32(page_indptr),
                         page_ids=i32(page_ids), fold_mode=i32(fold_mode),
                         fold_count=i32(fold_count), readout=i32(readout),
                         mask_word_indptr=None if mask_word_indptr is None else
                         np.ascontiguousarray(mask_word_indptr, dtype=np.int64))
        k = self.keep
        ptr = lambda a: None if a is None else a.ctypes.data
        self.c = abi.pie_fwd_meta(
            int(k["kv_len"].shape[0]), int(k["positions"].shape[0]), ptr(k["row_indptr"]),
            ptr(k["positions"]), ptr(k["slots"]), ptr(k["kv_len"]), ptr(k["page_indptr"]),
            ptr(k["page_ids"]), int(num_pool_pages), ptr(k["fold_mode"]), ptr(k["fold_count"]),
            ptr(k["mask_word_indptr"]), ptr(k["readout"]),
            0 if k["readout"] is None else int(k["readout"].shape[0]))


def make_meta(p, num_pool_pages: int, page_ids=None) -> _HostMeta:
    """From any object with the pass fields (row_indptr, positions, slots,
    kv_len, page_indptr, page_ids, fold_mode, fold_count, mask_word_indptr,
    readout)."""
    return _HostMeta(p.row_indptr, p.positions, p.slots, p.kv_len, p.page_indptr,
                     p.page_ids if page_ids is None else page_ids, num_pool_pages, p.fold_mode,
                     p.fold_count, p.mask_word_indptr, p.readout)


def workspace_bytes(desc: abi.pie_fwd_desc, meta: _HostMeta) -> int:
    n = C.c_size_t(0)
    abi.check(abi.load().pie_fwd_workspace_bytes(C.byref(desc), C.byref(meta.c), C.byref(n)),
              "pie_fwd_workspace_bytes")
    return int(n.value)


def set_timing_events(start=None, stop=None) -> None:
    """Have later attend calls on this thread record two timing-enabled
    torch.cuda.Event objects right around their attention kernels, and later
    readout_topk calls around their stream kernel (pie_fwd_set_timing_events);
    no arguments turns it off."""
    for e in (start, stop):
        if e is not None and not e.cuda_event:
            e.record()  # the CUDA event is created at its first record
    abi.check(abi.load().pie_fwd_set_timing_events(start.cuda_event if start is not None else None,
                                                   stop.cuda_event if stop is not None else None),
              "pie_fwd_set_timing_events")


def forward(desc: abi.pie_fwd_desc, meta: _HostMeta, workspace, q, k, v, q_rot, k_pool, v_pool,
            frozen_len, mask_words=None, out_readout=None, lse_readout=None, out_all=None,
            lse_all=None, channel=None, status=None, stream=None) -> None:
    """pie_fwd_forward: plan, append, (mask), attend and fold of one pass in
    one native call; workspace: uint8 CUDA tensor of at least
    workspace_bytes(desc, meta), busy until the pass's kernels finish."""
    abi.check(abi.load().pie_fwd_forward(
        C.byref(desc), C.byref(meta.c), _ptr(workspace, "workspace"), workspace.numel(),
        _ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(q_rot, "q_rot"), _ptr(k_pool, "k_pool"),
        _ptr(v_pool, "v_pool"), _ptr(frozen_len, "frozen_len"),
        _ptr(mask_words, "mask_words", False), _ptr(out_readout, "out_readout", False),
        _ptr(lse_readout, "lse_readout", False), _ptr(out_all, "out_all", False),
        _ptr(lse_all, "lse_all", False), _ptr(channel, "channel", False),
        _ptr(status, "status", False), _stream(stream)), "pie_fwd_forward")


def decode_loop_workspace_bytes(desc: abi.pie_fwd_desc, num_lanes: int, max_pages_per_lane: int) -> int:
    n = C.c_size_t(0)
    abi.check(abi.load().pie_fwd_decode_loop_workspace_bytes(C.byref(desc), num_lanes,
                                                             max_pages_per_lane, C.byref(n)),
              "pie_fwd_decode_loop_workspace_bytes")
    return int(n.value)


def decode_loop(desc: abi.pie_fwd_desc, page_indptr, page_ids, max_pages_per_lane: int,
                frozen_len, q, k, v, q_rot, k_pool, v_pool, out, lse=None, status=None,
                workspace=None, stream=None, channel=None):
    """pie_fwd_decode_loop: q [steps, L, Hq, d], k/v [steps, L, Hkv, d], out
    like q; page_indptr / page_ids / frozen_len int32 CUDA tensors; channel:
    optional int32 CUDA tensor [steps, L] of per-step fold counts."""
    import torch
    steps, L = int(q.shape[0]), int(q.shape[1])
    if workspace is None:
        need = decode_loop_workspace_bytes(desc, L, max_pages_per_lane)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    abi.check(abi.load().pie_fwd_decode_loop(
        C.byref(desc), L, steps, _ptr(page_indptr, "page_indptr"), _ptr(page_ids, "page_ids"),
        int(k_pool.shape[0]), max_pages_per_lane, _ptr(frozen_len, "frozen_len"), _ptr(q, "q"),
        _ptr(k, "k"),
        _ptr(v, "v"), _ptr(q_rot, "q_rot"), _ptr(k_pool, "k_pool"), _ptr(v_pool, "v_pool"),
        _ptr(out, "out"), _ptr(lse, "lse", False), _ptr(channel, "channel", False),
        _ptr(workspace, "workspace"), workspace.numel(),
        _ptr(status, "status", False), _stream(stream)), "pie_fwd_decode_loop")


def readout_topk_workspace_bytes(dtype: int, rows: int, vocab: int, k: int) -> int:
    n = C.c_size_t(0)
    abi.check(abi.load().pie_fwd_readout_topk_workspace_bytes(dtype, rows, vocab, k, C.byref(n)),
              "pie_fwd_readout_topk_workspace_bytes")
    return int(n.value)


def readout_topk(logits, k: int, ids, probs, z=None, lse=None, workspace=None, stream=None):
    """pie_fwd_readout_topk on a 2-D CUDA tensor of logits (float32 or
    bfloat16, rows of stride logits.stride(0)); ids int32 and probs float32
    [rows, k], z and lse float32 [rows] or None."""
    import torch
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be a 2-D tensor with unit column stride")
    if not logits.is_cuda:
        raise ValueError("logits must be a CUDA tensor")
    dtype = PIE_BF16 if logits.dtype == torch.bfloat16 else PIE_F32
    rows, vocab = logits.shape
    if workspace is None:
        need = readout_topk_workspace_bytes(dtype, rows, vocab, k)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=logits.device)
    abi.check(abi.load().pie_fwd_readout_topk(
        logits.data_ptr(), dtype, rows, vocab, logits.stride(0), k, _ptr(ids, "ids"),
        _ptr(probs, "probs"), _ptr(z, "z", False), _ptr(lse, "lse", False),
        _ptr(workspace, "workspace"), workspace.numel(), _stream(stream)), "pie_fwd_readout_topk")


def _ptr(t, what: str, required: bool = True):
    """Device address of a tensor; None becomes NULL (the C side decides
    whether the argument may be NULL)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return t.data_ptr()


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


class ForwardPlan:
    """One planned ForwardPass (pie_fwd_plan) and its three device steps.

    desc: pie_fwd_desc (see make_desc); meta: _HostMeta (see make_meta).
    workspace: optional uint8 CUDA tensor of at least workspace_bytes();
    allocated here when omitted.
    """

    def __init__(self, desc: abi.pie_fwd_desc, meta: _HostMeta, workspace=None, stream=None):
        import torch
        self.lib = abi.load()
        self.desc = desc
        self.meta = meta
        if workspace is None:
            need = workspace_bytes(desc, meta)
            workspace = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
        # a caller-supplied workspace that is too small is refused by the
        # planner itself (PIE_ENOSPACE)
        self.workspace = workspace
        h = C.c_void_p()
        abi.check(self.lib.pie_fwd_plan(C.byref(desc), C.byref(meta.c), _ptr(workspace, "workspace"),
                                        workspace.numel(), _stream(stream), C.byref(h)),
                  "pie_fwd_plan")
        self.handle = h
        self.num_readout = int(self.lib.pie_fwd_plan_num_readout(h))

    @classmethod
    def _adopt(cls, handle, desc: abi.pie_fwd_desc, workspace):
        """A ForwardPlan around a plan handle made elsewhere in the library
        (pie_batcher_plan_forward); it owns the handle from now on."""
        self = cls.__new__(cls)
        self.lib = abi.load()
        self.desc = desc
        self.meta = None
        self.workspace = workspace
        self.handle = handle
        self.num_readout = int(self.lib.pie_fwd_plan_num_readout(handle))
        return self

    def append_kv(self, q, k, v, q_rot, k_pool, v_pool, frozen_len, status=None, stream=None):
        abi.check(self.lib.pie_fwd_append_kv(
            self.handle, _ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(q_rot, "q_rot"),
            _ptr(k_pool, "k_pool"), _ptr(v_pool, "v_pool"), _ptr(frozen_len, "frozen_len"),
            _ptr(status, "status", False), _stream(stream)), "pie_fwd_append_kv")

    def set_mask(self, mask_words, stream=None):
        """pie_fwd_set_mask: build the pass's compacted mask lists once; later
        attend calls given the same mask_words tensor reuse them."""
        abi.check(self.lib.pie_fwd_set_mask(self.handle, _ptr(mask_words, "mask_words"),
                                            _stream(stream)), "pie_fwd_set_mask")

    def attend(self, q_rot, k_pool, v_pool, mask_words=None, out_readout=None, lse_readout=None,
               out_all=None, lse_all=None, status=None, stream=None):
        abi.check(self.lib.pie_fwd_attend(
            self.handle, _ptr(q_rot, "q_rot"), _ptr(k_pool, "k_pool"), _ptr(v_pool, "v_pool"),
            _ptr(mask_words, "mask_words", False), _ptr(out_readout, "out_readout", False),
            _ptr(lse_readout, "lse_readout", False), _ptr(out_all, "out_all", False),
            _ptr(lse_all, "lse_all", False), _ptr(status, "status", False), _stream(stream)),
            "pie_fwd_attend")

    def fold(self, frozen_len, channel=None, status=None, stream=None):
        abi.check(self.lib.pie_fwd_fold(
            self.handle, _ptr(frozen_len, "frozen_len"), _ptr(channel, "channel", False),
            _ptr(status, "status", False), _stream(stream)), "pie_fwd_fold")

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            self.lib.pie_fwd_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def adapter_workspace_bytes(row_indptr, max_rank: int = 16) -> int:
    """pie_fwd_adapter_workspace_bytes for host lanes (row_indptr [L+1])."""
    ri = np.ascontiguousarray(row_indptr, dtype=np.int32)
    n = C.c_size_t(0)
    abi.check(abi.load().pie_fwd_adapter_workspace_bytes(len(ri) - 1, ri.ctypes.data, max_rank,
                                                          C.byref(n)),
              "pie_fwd_adapter_workspace_bytes")
    return int(n.value)


class AdapterPlan:
    """Per-lane adapters of one pass (pie_fwd_adapter_plan): the lanes' rows
    cut into tiles, planned once and applied at any number of projection
    sites with apply().

    row_indptr [L+1] and adapter_of_lane [L] are host integer arrays
    (adapter -1: none); workspace is an optional uint8 CUDA tensor of at least
    adapter_workspace_bytes(), allocated here when omitted."""

    def __init__(self, row_indptr, adapter_of_lane, num_adapters: int, max_rank: int = 16,
                 workspace=None, stream=None):
        import torch
        self.lib = abi.load()
        ri = np.ascontiguousarray(row_indptr, dtype=np.int32)
        al = np.ascontiguousarray(adapter_of_lane, dtype=np.int32)
        if len(al) != len(ri) - 1:
            raise ValueError("adapter_of_lane needs one entry per lane")
        if workspace is None:
            need = adapter_workspace_bytes(ri, max_rank)
            workspace = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
        self.workspace = workspace
        h = C.c_void_p()
        abi.check(self.lib.pie_fwd_adapter_plan(
            len(al), ri.ctypes.data, al.ctypes.data, num_adapters, max_rank,
            _ptr(workspace, "workspace"), workspace.numel(), _stream(stream), C.byref(h)),
            "pie_fwd_adapter_plan")
        self.handle = h
        self.num_tiles = int(self.lib.pie_fwd_adapter_plan_num_tiles(h))
        self.num_groups = int(self.lib.pie_fwd_adapter_plan_num_groups(h))

    def apply(self, x, y, lora_a=None, lora_b=None, scale=None, ia3=None, status=None,
              stream=None):
        """y (bf16 [N, d_out], updated in place) += scale[a] B_a (A_a x), then
        scaled by ia3[a]; lora_a [n_ad, r, d_in], lora_b [n_ad, d_out, r],
        scale fp32 [n_ad], ia3 [n_ad, d_out] or None; lora_a None means rank 0
        (IA3 only)."""
        import torch
        if y.dtype != torch.bfloat16:
            raise ValueError("adapters are built for bfloat16")
        d_out = y.shape[1]
        rank = 0 if lora_a is None else lora_a.shape[1]
        d_in = x.shape[1] if x is not None else (lora_a.shape[2] if lora_a is not None else 64)
        abi.check(self.lib.pie_fwd_adapter_apply(
            self.handle, PIE_BF16, d_in, d_out, rank, _ptr(x, "x", False), _ptr(y, "y"),
            _ptr(lora_a, "lora_a", False), _ptr(lora_b, "lora_b", False),
            _ptr(scale, "scale", False), _ptr(ia3, "ia3", False), _ptr(status, "status", False),
            _stream(stream)), "pie_fwd_adapter_apply")

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            self.lib.pie_fwd_adapter_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Batcher:
    """Work-conserving dispatch of GPU-bound calls (pie_batcher_*): queues with
    priorities, calls with dependencies and read/write sets, one batch per
    dispatch() on a GPU-idle notification, complete() when it has run."""

    def __init__(self, ordered, max_calls: int, max_rows: int):
        self.lib = abi.load()
        flags = (C.c_uint8 * len(ordered))(*[1 if o else 0 for o in ordered])
        h = C.c_void_p()
        abi.check(self.lib.pie_batcher_create(len(ordered), flags, max_calls, max_rows,
                                              C.byref(h)), "pie_batcher_create")
        self.handle = h
        self.max_calls = max_calls
        self._calls = (C.c_int64 * max_calls)()
        self._lanes = (C.c_int32 * max_calls)()

    def add_queue(self, priority: int = 0) -> int:
        q = C.c_int32()
        abi.check(self.lib.pie_batcher_add_queue(self.handle, priority, C.byref(q)),
                  "pie_batcher_add_queue")
        return q.value

    def submit(self, queue: int, handler: int, rows: int, key: int = -1, deps=(), reads=(),
               writes=()) -> int:
        deps, reads, writes = (np.ascontiguousarray(x, dtype=np.int64).reshape(-1)
                               for x in (deps, reads, writes))
        cid = C.c_int64()
        abi.check(self.lib.pie_batcher_submit(
            self.handle, queue, handler, rows, key, deps.ctypes.data, deps.size,
            reads.ctypes.data, reads.size, writes.ctypes.data, writes.size, C.byref(cid)),
            "pie_batcher_submit")
        return cid.value

    def submit_many(self, queues, handlers, rows, keys, deps, reads, writes) -> range:
        """Enqueue len(queues) calls in one native call (pie_batcher_submit_many):
        per-call queue, handler, rows and key, and per-call lists of dependencies,
        read and write resource ids; returns the range of their ids."""
        n = len(queues)
        i32 = lambda x: np.ascontiguousarray(x, dtype=np.int32).reshape(-1)
        i64 = lambda x: np.ascontiguousarray(x, dtype=np.int64).reshape(-1)

        def flat(lists):
            sizes = [len(x) for x in lists]
            indptr = np.zeros(n + 1, dtype=np.int64)
            np.cumsum(sizes, out=indptr[1:])
            vals = i64(np.concatenate([i64(x) for x in lists])) if indptr[-1] else i64([])
            return indptr, vals
        q, h, r, k = i32(queues), i32(handlers), i64(rows), i64(keys)
        (di, dv), (ri, rv), (wi, wv) = flat(deps), flat(reads), flat(writes)
        first = C.c_int64()
        abi.check(self.lib.pie_batcher_submit_many(
            self.handle, n, q.ctypes.data, h.ctypes.data, r.ctypes.data, k.ctypes.data,
            di.ctypes.data, dv.ctypes.data, ri.ctypes.data, rv.ctypes.data, wi.ctypes.data,
            wv.ctypes.data, C.byref(first)), "pie_batcher_submit_many")
        return range(first.value, first.value + n)

    def dispatch(self, arrays: bool = False):
        """(handler, call ids, lanes) of the next batch, or None; with
        arrays=True the ids and lanes are numpy arrays (copies)."""
        n, h = C.c_int32(), C.c_int32()
        abi.check(self.lib.pie_batcher_dispatch(self.handle, self._calls, self._lanes,
                                                self.max_calls, C.byref(n), C.byref(h)),
                  "pie_batcher_dispatch")
        if n.value == 0:
            return None
        if arrays:
            return (h.value, np.ctypeslib.as_array(self._calls)[:n.value].copy(),
                    np.ctypeslib.as_array(self._lanes)[:n.value].copy())
        return h.value, list(self._calls[:n.value]), list(self._lanes[:n.value])

    def set_pages(self, key: int, pages) -> None:
        """pie_batcher_set_pages: working set `key`'s pool pages in slot order."""
        pages = np.ascontiguousarray(pages, dtype=np.int32).reshape(-1)
        abi.check(self.lib.pie_batcher_set_pages(self.handle, key, pages.ctypes.data, pages.size),
                  "pie_batcher_set_pages")

    def submit_forward(self, queues, keys, rows, first_slots, page_size: int,
                       handler: int = 0) -> range:
        """pie_batcher_submit_forward: forward calls on registered working
        sets, their read/write page sets derived natively; returns their ids."""
        q = np.ascontiguousarray(queues, dtype=np.int32).reshape(-1)
        k, r, f = (np.ascontiguousarray(x, dtype=np.int64).reshape(-1)
                   for x in (keys, rows, first_slots))
        first = C.c_int64()
        abi.check(self.lib.pie_batcher_submit_forward(
            self.handle, q.size, q.ctypes.data, handler, k.ctypes.data, r.ctypes.data,
            f.ctypes.data, page_size, C.byref(first)), "pie_batcher_submit_forward")
        return range(first.value, first.value + q.size)

    def plan_forward(self, ids, lanes, frozen, desc: abi.pie_fwd_desc, num_pool_pages: int,
                     workspace, stream=None):
        """pie_batcher_plan_forward: the pass of a dispatched forward batch,
        built and planned in one native call.  Returns (ForwardPlan, the working
        set of each lane, each call's first row, each lane's kv_len, rows).
        A workspace the planner refuses raises PieError(PIE_ENOSPACE)."""
        ids = np.ascontiguousarray(ids, dtype=np.int64).reshape(-1)
        lanes = np.ascontiguousarray(lanes, dtype=np.int32).reshape(-1)
        frozen = np.ascontiguousarray(frozen, dtype=np.int32).reshape(-1)
        n = ids.size
        bufs = getattr(self, "_pf", None)
        if bufs is None or bufs[0].size < n:
            bufs = self._pf = (np.zeros(max(n, 1), np.int64), np.zeros(max(n, 1), np.int32),
                               np.zeros(max(n, 1), np.int32))
        keys, first, kv = bufs
        h, nl, nr = C.c_void_p(), C.c_int32(), C.c_int32()
        abi.check(self.lib.pie_batcher_plan_forward(
            self.handle, ids.ctypes.data, lanes.ctypes.data, n, frozen.ctypes.data, frozen.size,
            C.byref(desc), num_pool_pages, _ptr(workspace, "workspace"), workspace.numel(),
            _stream(stream), C.byref(h), keys.ctypes.data, first.ctypes.data, kv.ctypes.data,
            C.byref(nl), C.byref(nr)), "pie_batcher_plan_forward")
        L = nl.value
        return (ForwardPlan._adopt(h, desc, workspace), keys[:L], first[:n], kv[:L], nr.value)

    def forward_pass(self, ids, lanes, frozen):
        """pie_batcher_forward_pass: the pass fields (as make_meta takes them)
        of a dispatched forward batch, the working set of each lane and each
        call's first row.  frozen: int32 array of frozen lengths by key.  The
        returned arrays are views of buffers reused by the next call."""
        ids = np.ascontiguousarray(ids, dtype=np.int64).reshape(-1)
        lanes = np.ascontiguousarray(lanes, dtype=np.int32).reshape(-1)
        frozen = np.ascontiguousarray(frozen, dtype=np.int32).reshape(-1)
        n = ids.size
        nl, nr, npg = C.c_int32(), C.c_int32(), C.c_int64()
        for _ in range(2):
            bufs = getattr(self, "_fp", None)
            if bufs is None:
                bufs = self._fp = dict(L=0, N=0, P=0)
            if bufs["L"] >= max(n, 1) and bufs["N"] >= max(nr.value, 1) and \
                    bufs["P"] >= max(npg.value, 1):
                pass
            else:
                L, N, P = max(n, 1, bufs["L"]), max(nr.value, 1, bufs["N"]), max(npg.value, 1, bufs["P"])
                bufs.update(L=L, N=N, P=P, row_indptr=np.zeros(L + 1, np.int32),
                            positions=np.zeros(N, np.int32), kv_len=np.zeros(L, np.int32),
                            page_indptr=np.zeros(L + 1, np.int32), page_ids=np.zeros(P, np.int32),
                            lane_keys=np.zeros(L, np.int64), first_row=np.zeros(L, np.int32),
                            fold_mode=np.full(L, abi.PIE_FOLD_ALL, np.int32),
                            fold_count=np.zeros(L, np.int32))
            rc = self.lib.pie_batcher_forward_pass(
                self.handle, ids.ctypes.data, lanes.ctypes.data, n, frozen.ctypes.data,
                frozen.size, bufs["L"], bufs["N"], bufs["P"], bufs["row_indptr"].ctypes.data,
                bufs["positions"].ctypes.data, bufs["kv_len"].ctypes.data,
                bufs["page_indptr"].ctypes.data, bufs["page_ids"].ctypes.data,
                bufs["lane_keys"].ctypes.data, bufs["first_row"].ctypes.data, C.byref(nl),
                C.byref(nr), C.byref(npg))
            if rc != abi.PIE_ENOSPACE:
                break
        abi.check(rc, "pie_batcher_forward_pass")
        L, N, P = nl.value, nr.value, int(npg.value)
        pos = bufs["positions"][:N]
        p = types.SimpleNamespace(
            row_indptr=bufs["row_indptr"][:L + 1], positions=pos, slots=pos,
            kv_len=bufs["kv_len"][:L], page_indptr=bufs["page_indptr"][:L + 1],
            page_ids=bufs["page_ids"][:P], fold_mode=bufs["fold_mode"][:L],
            fold_count=bufs["fold_count"][:L], mask_word_indptr=None, readout=None)
        return p, bufs["lane_keys"][:L], bufs["first_row"][:n]

    def complete(self, ids):
        ids = np.ascontiguousarray(ids, dtype=np.int64).reshape(-1)
        abi.check(self.lib.pie_batcher_complete(self.handle, ids.ctypes.data, ids.size),
                  "pie_batcher_complete")

    def counts(self):
        a, b = C.c_int64(), C.c_int64()
        abi.check(self.lib.pie_batcher_counts(self.handle, C.byref(a), C.byref(b)),
                  "pie_batcher_counts")
        return a.value, b.value

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            self.lib.pie_batcher_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
