"""The no-allocation decode attention entry point against the planned path.

pie_fwd_decode_attend_noalloc serves callers that cannot allocate device
memory when they launch attention (a foreign memory manager with a fixed
device budget, or a host path that must not take the allocator's locks):
it takes its scratch from a static device array of the library instead of a
caller workspace.  This test calls it through the C ABI twice in a row, on
two different decode batches, and checks each output against the output of
the existing entry points (pie_fwd_plan / pie_fwd_append_kv /
pie_fwd_attend) on the same inputs, within the attention tolerance the
parity tests use.  It also checks that a call needing more scratch than the
array holds is refused.  This file is collected last so that a failure here
never hides another test's result.
"""
import ctypes as C

import numpy as np
import pytest

import workloads as W
from tests.parity import OUT_TOL

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _planned_and_noalloc(sc):
    from programmable_paged_kv_gb300 import ForwardPlan, abi, make_desc, make_meta, runner
    lib = abi.load()
    d = sc.desc
    p = sc.passes[0]
    desc = make_desc(d)
    pools = runner.DevicePools(sc)
    frozen = torch.from_numpy(sc.frozen_len0.astype(np.int32)).cuda()
    tdt = torch.bfloat16 if d.dtype == W.BF16 else torch.float32
    L, Hq, D = p.num_lanes, d.num_q_heads, d.head_dim
    q_rot = torch.empty((L, Hq, D), dtype=tdt, device="cuda")
    plan = ForwardPlan(desc, make_meta(p, sc.num_pool_pages))
    plan.append_kv(runner.to_device(p.q, d.dtype), runner.to_device(p.k, d.dtype),
                   runner.to_device(p.v, d.dtype), q_rot, pools.k, pools.v, frozen)
    ref = torch.empty((L, Hq, D), dtype=tdt, device="cuda")
    ref_lse = torch.empty((L, Hq), dtype=torch.float32, device="cuda")
    plan.attend(q_rot, pools.k, pools.v, None, ref, ref_lse)

    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
    slots, kv_len = dev(p.slots), dev(p.kv_len)
    page_indptr, page_ids = dev(p.page_indptr), dev(p.page_ids)
    out = torch.full((L, Hq, D), float("nan"), dtype=tdt, device="cuda")
    lse = torch.full((L, Hq), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.pie_fwd_decode_attend_noalloc(
        C.byref(desc), L, int(p.kv_len.max()), slots.data_ptr(), kv_len.data_ptr(),
        page_indptr.data_ptr(), page_ids.data_ptr(), q_rot.data_ptr(), pools.k.data_ptr(),
        pools.v.data_ptr(), out.data_ptr(), lse.data_ptr(), status.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert rc == abi.PIE_OK, lib.pie_fwd_last_error()
    torch.cuda.synchronize()
    plan.close()
    return ref, ref_lse, out, lse, int(status.item())


def test_no_alloc_decode_matches_planned_attend_twice_in_a_row():
    first = W.decode_batch(5, lanes=9, c_lo=1, c_hi=700, num_pool_pages=1024)
    second = W.decode_batch(6, lanes=64, c_lo=512, c_hi=4096, num_pool_pages=16384)
    mx, mean = OUT_TOL[W.BF16]
    for sc in (first, second):
        ref, ref_lse, out, lse, status = _planned_and_noalloc(sc)
        assert status == 0
        err = (out.float() - ref.float()).abs()
        assert torch.isfinite(out.float()).all()
        assert err.max().item() <= mx and err.mean().item() <= mean
        assert (lse - ref_lse).abs().max().item() <= 1e-3


def test_no_alloc_refuses_scratch_overflow():
    from programmable_paged_kv_gb300 import abi, make_desc
    lib = abi.load()
    desc = make_desc(W.Desc(32, 8, 128, 16, W.BF16))
    one = torch.zeros(8, dtype=torch.int32, device="cuda")
    rc = lib.pie_fwd_decode_attend_noalloc(
        C.byref(desc), 256, 1 << 20, one.data_ptr(), one.data_ptr(), one.data_ptr(),
        one.data_ptr(), one.data_ptr(), one.data_ptr(), one.data_ptr(), one.data_ptr(), None,
        None, torch.cuda.current_stream().cuda_stream)
    assert rc == abi.PIE_ERANGE
    assert b"static scratch" in lib.pie_fwd_last_error()
