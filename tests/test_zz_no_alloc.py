"""The no-allocation decode attention entry point against the planned path.

pie_fwd_decode_attend_noalloc serves callers that cannot allocate device
memory when they launch attention (a foreign memory manager with a fixed
device budget, or a host path that must not take the allocator's locks):
it takes its scratch from a static device array of the library instead of a
caller workspace.  These tests call it through the C ABI and check its
output against the existing entry points (pie_fwd_plan / pie_fwd_append_kv /
pie_fwd_attend) on the same inputs, within the attention tolerance the
parity tests use:
  * two calls in a row on two different decode batches, small then large;
  * 200 calls queued back to back on one stream with no host wait between
    them, their lane counts and kv lengths changing from call to call
    (large after small and small after large, same shape with other
    lengths), every output checked: a call must never see the work items or
    partial states an earlier call left in the shared scratch;
  * a call whose max_kv_len is below some lane's kv_len: the status bit is
    set and the output is attention over the first max_kv_len slots, as the
    oracle computes it;
  * a call needing more scratch than the array holds is refused;
  * device page tables are checked: a kv_len past a lane's pages is cut, a
    page id outside the pool is not read, and the status says so.
This file is collected last so that a failure here never hides another
test's result.
"""
import ctypes as C

import numpy as np
import pytest

import workloads as W
from tests.parity import LSE_TOL, OUT_TOL

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

PIE_STATUS_NOALLOC_TRUNC = 32


def _dev32(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()


def _setup(sc):
    """Pools and rotated queries of the scenario's first pass (its K/V
    appended through the planned path)."""
    from programmable_paged_kv_gb300 import ForwardPlan, make_desc, make_meta, runner
    d = sc.desc
    p = sc.passes[0]
    desc = make_desc(d)
    pools = runner.DevicePools(sc)
    frozen = torch.from_numpy(sc.frozen_len0.astype(np.int32)).cuda()
    tdt = torch.bfloat16 if d.dtype == W.BF16 else torch.float32
    q_rot = torch.empty((p.num_lanes, d.num_q_heads, d.head_dim), dtype=tdt, device="cuda")
    plan = ForwardPlan(desc, make_meta(p, sc.num_pool_pages))
    plan.append_kv(runner.to_device(p.q, d.dtype), runner.to_device(p.k, d.dtype),
                   runner.to_device(p.v, d.dtype), q_rot, pools.k, pools.v, frozen)
    torch.cuda.synchronize()
    plan.close()
    return desc, pools, q_rot, tdt


def _planned(sc, desc, pools, q_rot, tdt, kv_len, slots):
    """pie_fwd_plan + pie_fwd_attend over the given kv lengths and slots."""
    from programmable_paged_kv_gb300 import ForwardPlan, make_meta
    p = sc.passes[0]
    L = p.num_lanes
    meta_p = W.Pass(p.row_indptr, p.positions, np.asarray(slots, np.int32),
                    np.asarray(kv_len, np.int32), p.page_indptr, p.page_ids, p.fold_mode,
                    p.fold_count, p.q, p.k, p.v)
    plan = ForwardPlan(desc, make_meta(meta_p, sc.num_pool_pages))
    ref = torch.empty((L, sc.desc.num_q_heads, sc.desc.head_dim), dtype=tdt, device="cuda")
    ref_lse = torch.empty((L, sc.desc.num_q_heads), dtype=torch.float32, device="cuda")
    plan.attend(q_rot, pools.k, pools.v, None, ref, ref_lse)
    torch.cuda.synchronize()
    plan.close()
    return ref, ref_lse


def _noalloc(lib, desc, n, max_kv, slots_d, kv_d, pind_d, pids_d, q_rot, pools, out, lse,
             status):
    return lib.pie_fwd_decode_attend_noalloc(
        C.byref(desc), n, int(max_kv), slots_d.data_ptr(), kv_d.data_ptr(), pind_d.data_ptr(),
        pids_d.data_ptr(), int(pools.k.shape[0]), q_rot.data_ptr(), pools.k.data_ptr(),
        pools.v.data_ptr(),
        out.data_ptr(), lse.data_ptr(), status.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def _close(out, lse, ref, ref_lse, dtype=W.BF16):
    mx, mean = OUT_TOL[dtype]
    assert torch.isfinite(out.float()).all()
    err = (out.float() - ref.float()).abs()
    assert err.max().item() <= mx and err.mean().item() <= mean, (err.max().item(),
                                                                  err.mean().item())
    assert (lse - ref_lse).abs().max().item() <= LSE_TOL[dtype]


def test_no_alloc_decode_matches_planned_attend_twice_in_a_row():
    from programmable_paged_kv_gb300 import abi
    lib = abi.load()
    first = W.decode_batch(5, lanes=9, c_lo=1, c_hi=700, num_pool_pages=1024)
    second = W.decode_batch(6, lanes=64, c_lo=512, c_hi=4096, num_pool_pages=16384)
    for sc in (first, second):
        p = sc.passes[0]
        desc, pools, q_rot, tdt = _setup(sc)
        ref, ref_lse = _planned(sc, desc, pools, q_rot, tdt, p.kv_len, p.slots)
        L = p.num_lanes
        out = torch.full_like(ref, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = _noalloc(lib, desc, L, p.kv_len.max(), _dev32(p.slots), _dev32(p.kv_len),
                      _dev32(p.page_indptr), _dev32(p.page_ids), q_rot, pools, out, lse, status)
        assert rc == abi.PIE_OK, lib.pie_fwd_last_error()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        _close(out, lse, ref, ref_lse)


def test_no_alloc_200_calls_back_to_back_with_changing_shapes():
    """Calls queued with no host wait between them; lane counts and kv
    lengths change every call, so each call's work items, combine entries
    and partial states overwrite a differently shaped set left by the call
    before (more lanes and chunks before fewer, and fewer before more)."""
    from programmable_paged_kv_gb300 import abi
    lib = abi.load()
    sc = W.decode_batch(11, lanes=64, c_lo=16, c_hi=4096, num_pool_pages=20000)
    p = sc.passes[0]
    desc, pools, q_rot, tdt = _setup(sc)
    L = p.num_lanes
    cap = p.kv_len  # every lane's K/V holds finite values in slots [0, C + 1)
    rng = np.random.default_rng(7)
    # eight variants of the lanes' lengths; kv_len in [1, cap], own slot last
    variants = []
    for v in range(8):
        lo = 1 if v % 2 else max(1, int(cap.min()) // 2)
        kv = np.minimum(cap, rng.integers(lo, cap + 1)).astype(np.int32)
        kv = np.maximum(kv, 1)
        slots = (kv - 1).astype(np.int32)
        ref, ref_lse = _planned(sc, desc, pools, q_rot, tdt, kv, slots)
        variants.append((_dev32(kv), _dev32(slots), int(kv.max()), ref, ref_lse))
    pind, pids = _dev32(p.page_indptr), _dev32(p.page_ids)
    calls = 200
    order = rng.integers(0, len(variants), size=calls)
    lanes = rng.choice([64, 3, 40, 17, 64, 1, 29, 64], size=calls)
    Hq, D = sc.desc.num_q_heads, sc.desc.head_dim
    outs = torch.full((calls, L, Hq, D), float("nan"), dtype=tdt, device="cuda")
    lses = torch.full((calls, L, Hq), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for i in range(calls):
        kv_d, slots_d, mx, _, _ = variants[order[i]]
        n = int(lanes[i])
        rc = _noalloc(lib, desc, n, mx, slots_d, kv_d, pind, pids, q_rot, pools, outs[i],
                      lses[i], status)
        assert rc == abi.PIE_OK, lib.pie_fwd_last_error()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for i in range(calls):
        _, _, _, ref, ref_lse = variants[order[i]]
        n = int(lanes[i])
        _close(outs[i, :n], lses[i, :n], ref[:n], ref_lse[:n])
        # rows past the call's lanes are not written
        assert torch.isnan(lses[i, n:]).all()


def test_no_alloc_truncates_to_max_kv_len_like_the_oracle():
    """max_kv_len below some lanes' kv_len: those lanes attend over their
    first max_kv_len slots, PIE_STATUS_NOALLOC_TRUNC is set; the result is
    the oracle's attention with kv_len cut to max_kv_len."""
    import oracle as O
    from programmable_paged_kv_gb300 import abi, runner
    lib = abi.load()
    sc = W.decode_batch(12, lanes=12, c_lo=100, c_hi=1500, num_pool_pages=2048)
    p = sc.passes[0]
    desc, pools, q_rot, tdt = _setup(sc)
    L = p.num_lanes
    max_kv = 700
    assert (p.kv_len > max_kv).any() and (p.kv_len <= max_kv).any()
    out = torch.full((L, sc.desc.num_q_heads, sc.desc.head_dim), float("nan"), dtype=tdt,
                     device="cuda")
    lse = torch.full((L, sc.desc.num_q_heads), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = _noalloc(lib, desc, L, max_kv, _dev32(p.slots), _dev32(p.kv_len), _dev32(p.page_indptr),
                  _dev32(p.page_ids), q_rot, pools, out, lse, status)
    assert rc == abi.PIE_OK, lib.pie_fwd_last_error()
    torch.cuda.synchronize()
    assert int(status.item()) & PIE_STATUS_NOALLOC_TRUNC
    # the oracle: the same pass with kv_len cut to max_kv_len (the row's own
    # slot then lies past the cut and is not visible)
    cut = W.Pass(p.row_indptr, p.positions, p.slots, np.minimum(p.kv_len, max_kv).astype(np.int32),
                 p.page_indptr, p.page_ids, p.fold_mode, p.fold_count, p.q, p.k, p.v)
    k0, v0, fz = sc.k_init.copy(), sc.v_init.copy(), sc.frozen_len0.copy()
    r = O.run_pass(sc.desc, cut, k0, v0, fz, page_ids=sc.compact_page_ids(p.page_ids),
                   num_threads=8, do_fold=False)
    assert r["err"] == O.OK
    got = W.storage_to_f32(runner.to_host(out, sc.desc.dtype), sc.desc.dtype).astype(np.float64)
    err = np.abs(got - r["out"])
    mx, mean = OUT_TOL[W.BF16]
    assert err.max() <= mx and err.mean() <= mean
    assert np.abs(lse.cpu().numpy() - r["lse"]).max() <= LSE_TOL[W.BF16]


def test_no_alloc_refuses_scratch_overflow():
    from programmable_paged_kv_gb300 import abi, make_desc
    lib = abi.load()
    desc = make_desc(W.Desc(32, 8, 128, 16, W.BF16))
    one = torch.zeros(8, dtype=torch.int32, device="cuda")
    rc = lib.pie_fwd_decode_attend_noalloc(
        C.byref(desc), 256, 1 << 20, one.data_ptr(), one.data_ptr(), one.data_ptr(),
        one.data_ptr(), 1, one.data_ptr(), one.data_ptr(), one.data_ptr(), one.data_ptr(), None,
        None, torch.cuda.current_stream().cuda_stream)
    assert rc == abi.PIE_ERANGE
    assert b"static scratch" in lib.pie_fwd_last_error()


def test_no_alloc_checks_device_page_tables():
    """The page table is device data: a lane whose kv_len runs past its pages
    is cut to them, and a page id outside the pool is not read; both set
    PIE_STATUS_BOUNDS, and every other lane still gets the planned path's
    output."""
    from programmable_paged_kv_gb300 import abi
    lib = abi.load()
    sc = W.decode_batch(13, lanes=10, c_lo=100, c_hi=900, num_pool_pages=2048)
    p = sc.passes[0]
    desc, pools, q_rot, tdt = _setup(sc)
    ref, ref_lse = _planned(sc, desc, pools, q_rot, tdt, p.kv_len, p.slots)
    L = p.num_lanes
    kv_bad = p.kv_len.copy()
    slots_bad = p.slots.copy()
    cap = np.diff(p.page_indptr) * sc.desc.page_size
    kv_bad[2] = cap[2] + 500         # past lane 2's pages
    slots_bad[2] = cap[2] + 499
    ids_bad = p.page_ids.copy()
    ids_bad[p.page_indptr[5] + 1] = 1 << 30   # outside the pool
    ids_bad[p.page_indptr[7]] = -3
    out = torch.full_like(ref, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = _noalloc(lib, desc, L, int(kv_bad.max()), _dev32(slots_bad), _dev32(kv_bad),
                  _dev32(p.page_indptr), _dev32(ids_bad), q_rot, pools, out, lse, status)
    assert rc == abi.PIE_OK, lib.pie_fwd_last_error()
    torch.cuda.synchronize()
    assert int(status.item()) & 4  # PIE_STATUS_BOUNDS
    good = [l for l in range(L) if l not in (2, 5, 7)]
    _close(out[good], lse[good], ref[good], ref_lse[good])
