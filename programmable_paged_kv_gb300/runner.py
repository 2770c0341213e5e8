"""Drive a sequence of ForwardPasses (a `workloads.Scenario`) through the C
ABI on one GPU and bring the results back to the host.

Everything on the path runs in libpie_fwd.so; this module only allocates the
device tensors, uploads the seeded inputs, calls plan / append_kv / attend /
fold in order on the current stream, and plays the epilogue's part of
writing the accepted counts into the fold channel.
"""
from __future__ import annotations

import numpy as np

from . import ForwardPlan, make_desc, make_meta

_TORCH_DT = None


def torch_storage_dtype(dtype: int):
    import torch
    return torch.float32 if dtype == 0 else torch.int16


def to_device(a: np.ndarray, dtype: int):
    """Storage array (float32 or bf16 bit patterns) -> CUDA tensor of the
    pass dtype (float32 or bfloat16), bit for bit."""
    import torch
    if dtype == 0:
        return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
    return t.view(torch.bfloat16)


def to_host(t, dtype: int) -> np.ndarray:
    """CUDA tensor of the pass dtype -> storage array (bits preserved)."""
    import torch
    if dtype == 0:
        return t.detach().float().cpu().numpy()
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class DevicePools:
    """Full-size K/V pools on the device, canary-filled, with the scenario's
    initial pages written at their physical ids.  A scenario built without
    its cached contents (workloads.geometry_only) gets its pages filled here
    with N(0,1) values from a seeded device generator instead."""

    def __init__(self, sc, seed: int = 0):
        import torch
        d = sc.desc
        shape = (sc.num_pool_pages, d.num_kv_heads, d.page_size, d.head_dim)
        if d.dtype == 0:
            self.k = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
            self.k.view(torch.int32).fill_(-1)
        else:
            self.k = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
            self.k.view(torch.int16).fill_(-1)
        self.v = self.k.clone()
        idx = torch.from_numpy(sc.pool_pages.astype(np.int64)).cuda()
        if sc.k_init is None:
            g = torch.Generator(device="cuda")
            g.manual_seed(seed)
            tdt = torch.float32 if d.dtype == 0 else torch.bfloat16
            for t in (self.k, self.v):
                for i in range(0, idx.numel(), 4096):
                    part = idx[i:i + 4096]
                    t.index_copy_(0, part, torch.randn((part.numel(),) + shape[1:], generator=g,
                                                       device="cuda").to(tdt))
        else:
            self.k.index_copy_(0, idx, to_device(sc.k_init, d.dtype))
            self.v.index_copy_(0, idx, to_device(sc.v_init, d.dtype))
        self.used = idx


def run_scenario(sc, want_all: bool = True, status_per_pass: bool = True, one_call: bool = False):
    """Run every pass of `sc`; returns (k_used, v_used, frozen, results) where
    k_used/v_used are the pool pages listed in sc.pool_pages (storage arrays)
    and results[i] holds q_rot, out_all, lse_all, out_readout, lse_readout
    and status of pass i.  one_call: each pass through pie_fwd_forward
    instead of plan / append_kv / attend / fold."""
    import torch
    d = sc.desc
    desc = make_desc(d)
    pools = DevicePools(sc)
    frozen = torch.from_numpy(sc.frozen_len0.astype(np.int32)).cuda()
    results = []
    for p in sc.passes:
        meta = make_meta(p, sc.num_pool_pages)
        plan = ForwardPlan(desc, meta)
        if one_call:  # only its readout count is used; the pass plans itself
            R = plan.num_readout
            plan.close()
        N, Hq, D = p.num_rows, d.num_q_heads, d.head_dim
        tdt = torch.float32 if d.dtype == 0 else torch.bfloat16
        q = to_device(p.q, d.dtype)
        k = to_device(p.k, d.dtype)
        v = to_device(p.v, d.dtype)
        q_rot = torch.empty((N, Hq, D), dtype=tdt, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        if not one_call:
            plan.append_kv(q, k, v, q_rot, pools.k, pools.v, frozen, status)
            R = plan.num_readout
        out_ro = torch.empty((R, Hq, D), dtype=tdt, device="cuda")
        lse_ro = torch.empty((R, Hq), dtype=torch.float32, device="cuda")
        out_all = torch.empty((N, Hq, D), dtype=tdt, device="cuda") if want_all else None
        lse_all = torch.empty((N, Hq), dtype=torch.float32, device="cuda") if want_all else None
        mw = None
        if p.mask_words is not None:
            mw = torch.from_numpy(p.mask_words.view(np.int32)).cuda()
        chan = None
        if p.channel is not None:
            # the epilogue's write of the accepted counts, ordered on the stream
            chan = torch.from_numpy(p.channel.astype(np.int32)).cuda()
        if one_call:
            from . import forward, workspace_bytes
            ws = torch.empty(workspace_bytes(desc, meta) + 256, dtype=torch.uint8, device="cuda")
            forward(desc, meta, ws, q, k, v, q_rot, pools.k, pools.v, frozen, mw, out_ro, lse_ro,
                    out_all, lse_all, chan, status)
        else:
            plan.attend(q_rot, pools.k, pools.v, mw, out_ro, lse_ro, out_all, lse_all, status)
            plan.fold(frozen, chan, status)
        torch.cuda.synchronize()
        res = dict(q_rot=to_host(q_rot, d.dtype), out_readout=to_host(out_ro, d.dtype),
                   lse_readout=lse_ro.cpu().numpy(), status=int(status.item()) & 0xFFFFFFFF)
        if want_all:
            res["out_all"] = to_host(out_all, d.dtype)
            res["lse_all"] = lse_all.cpu().numpy()
        results.append(res)
        if not one_call:
            plan.close()
    k_used = to_host(pools.k.index_select(0, pools.used), d.dtype)
    v_used = to_host(pools.v.index_select(0, pools.used), d.dtype)
    untouched_ok = _untouched_is_canary(pools, d.dtype)
    return k_used, v_used, frozen.cpu().numpy(), results, untouched_ok


def _untouched_is_canary(pools, dtype) -> bool:
    """True iff every page outside the scenario's pages still holds the canary."""
    import torch
    keep = torch.ones(pools.k.shape[0], dtype=torch.bool, device="cuda")
    keep[pools.used] = False
    it = torch.int32 if dtype == 0 else torch.int16
    for t in (pools.k, pools.v):
        bits = t.view(it)[keep]
        if bits.numel() and not bool((bits == -1).all()):
            return False
    return True
