"""The bounded-wait failure path, run without faulting or hanging the GPU.

Every wait of the split-KV attention kernel gives up after a time limit and
sets PIE_STATUS_TIMEOUT.  pie_fwd_test_wait_expiry makes that happen on
purpose and safely: the kernel's producer warp stops before a chosen stage of
every work item, so no copy of that stage (or of a later one) is ever in
flight, and the compute warps' wait for it runs out after a short limit.  The
test checks that the status word says so, that the call returns, and that
the same plan then attends correctly once the hook is off (the context is
intact).
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests.parity import compare_scenario

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

PIE_STATUS_TIMEOUT = 16


def test_expired_wait_sets_timeout_and_the_context_stays_usable():
    from programmable_paged_kv_gb300 import ForwardPlan, abi, make_desc, make_meta, runner
    lib = abi.load()
    sc = W.decode_batch(21, lanes=12, c_lo=200, c_hi=1200, num_pool_pages=1024)
    d, p = sc.desc, sc.passes[0]
    desc = make_desc(d)
    pools = runner.DevicePools(sc)
    frozen = torch.from_numpy(sc.frozen_len0.astype(np.int32)).cuda()
    N, Hq, D = p.num_rows, d.num_q_heads, d.head_dim
    q_rot = torch.empty((N, Hq, D), dtype=torch.bfloat16, device="cuda")
    plan = ForwardPlan(desc, make_meta(p, sc.num_pool_pages))
    plan.append_kv(*(runner.to_device(x, d.dtype) for x in (p.q, p.k, p.v)), q_rot, pools.k,
                   pools.v, frozen)
    out = torch.empty((plan.num_readout, Hq, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((plan.num_readout, Hq), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.pie_fwd_test_wait_expiry(1, 300) == abi.PIE_OK  # stop before stage 1, 300 us
    try:
        plan.attend(q_rot, pools.k, pools.v, None, out, lse, None, None, status)
        torch.cuda.synchronize()
    finally:
        assert lib.pie_fwd_test_wait_expiry(-1, 0) == abi.PIE_OK
    assert int(status.item()) & PIE_STATUS_TIMEOUT
    # the hook off: the same plan, pools and queries give the oracle's result
    status.zero_()
    out_all = torch.empty((N, Hq, D), dtype=torch.bfloat16, device="cuda")
    lse_all = torch.empty((N, Hq), dtype=torch.float32, device="cuda")
    plan.attend(q_rot, pools.k, pools.v, None, out, lse, out_all, lse_all, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    orc = O.run_scenario(sc, num_threads=4)
    from tests.parity import assert_out_close, assert_lse_close
    assert_out_close(runner.to_host(out_all, d.dtype), orc[3][0]["out"], d.dtype, "out")
    assert_lse_close(lse_all.cpu().numpy(), orc[3][0]["lse"], d.dtype, "lse")
    plan.close()


def test_expired_wait_on_a_masked_pass_with_several_items_per_cta():
    # masked decode rows walk their compacted visible-slot lists, two work
    # items per CTA: after the first item's wait runs out the CTA's warps
    # still take every barrier of its later items, so the call returns
    from programmable_paged_kv_gb300 import ForwardPlan, abi, make_desc, make_meta, runner
    lib = abi.load()
    sc = W.small("masked_decode_window", 1)
    d, p = sc.desc, sc.passes[0]
    desc = make_desc(d)
    pools = runner.DevicePools(sc)
    frozen = torch.from_numpy(sc.frozen_len0.astype(np.int32)).cuda()
    N, Hq, D = p.num_rows, d.num_q_heads, d.head_dim
    q_rot = torch.empty((N, Hq, D), dtype=torch.bfloat16, device="cuda")
    plan = ForwardPlan(desc, make_meta(p, sc.num_pool_pages))
    plan.append_kv(*(runner.to_device(x, d.dtype) for x in (p.q, p.k, p.v)), q_rot, pools.k,
                   pools.v, frozen)
    mw = torch.from_numpy(p.mask_words.view(np.int32)).cuda()
    out = torch.empty((plan.num_readout, Hq, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((plan.num_readout, Hq), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.pie_fwd_test_wait_expiry(1, 300) == abi.PIE_OK
    try:
        plan.attend(q_rot, pools.k, pools.v, mw, out, lse, None, None, status)
        torch.cuda.synchronize()
    finally:
        assert lib.pie_fwd_test_wait_expiry(-1, 0) == abi.PIE_OK
    assert int(status.item()) & PIE_STATUS_TIMEOUT
    status.zero_()
    out_all = torch.empty((N, Hq, D), dtype=torch.bfloat16, device="cuda")
    lse_all = torch.empty((N, Hq), dtype=torch.float32, device="cuda")
    plan.attend(q_rot, pools.k, pools.v, mw, out, lse, out_all, lse_all, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    orc = O.run_scenario(sc, num_threads=4)
    from tests.parity import assert_out_close, assert_lse_close
    assert_out_close(runner.to_host(out_all, d.dtype), orc[3][0]["out"], d.dtype, "out")
    assert_lse_close(lse_all.cpu().numpy(), orc[3][0]["lse"], d.dtype, "lse")
    plan.close()


def test_hook_arguments_are_checked():
    from programmable_paged_kv_gb300 import abi
    lib = abi.load()
    assert lib.pie_fwd_test_wait_expiry(-2, 10) == abi.PIE_EINVAL
    assert lib.pie_fwd_test_wait_expiry(0, 0) == abi.PIE_EINVAL
    assert lib.pie_fwd_test_wait_expiry(-1, 0) == abi.PIE_OK
