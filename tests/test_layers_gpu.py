"""One plan serves every layer of a pass ("The forward pass": the plan and its
mask belong to the ForwardPass; each attention layer calls attend with its own
queries and caches).  The split-KV kernel of a plain pass runs as a persistent
grid that takes its work items from a counter in the plan's workspace, which
the kernel's last CTA sets back to zero; so repeated attend calls on one plan
must each compute their own result: a call with other queries differs and
equals a fresh plan's result bit for bit, and repeating the first call
reproduces it bit for bit."""
import numpy as np
import pytest

import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from programmable_paged_kv_gb300 import build
    build()


def test_attend_repeated_on_one_plan_computes_each_call():
    from programmable_paged_kv_gb300 import ForwardPlan, make_desc, make_meta, runner
    sc = W.decode_batch(5, lanes=16, c_lo=100, c_hi=2000, num_pool_pages=2048)
    d, p = sc.desc, sc.passes[0]
    desc, meta = make_desc(d), make_meta(p, sc.num_pool_pages)
    pools = runner.DevicePools(sc)
    frozen = torch.from_numpy(sc.frozen_len0.astype(np.int32)).cuda()
    N, Hq, D = p.num_rows, d.num_q_heads, d.head_dim
    q_rot1 = torch.empty((N, Hq, D), dtype=torch.bfloat16, device="cuda")
    plan = ForwardPlan(desc, meta)
    plan.append_kv(*(runner.to_device(x, d.dtype) for x in (p.q, p.k, p.v)), q_rot1, pools.k,
                   pools.v, frozen)
    q_rot2 = (q_rot1.float() * -0.75).to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def attend(pl, q):
        out = torch.empty((N, Hq, D), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((N, Hq), dtype=torch.float32, device="cuda")
        pl.attend(q, pools.k, pools.v, None, None, None, out, lse, status)
        return out, lse

    o1, l1 = attend(plan, q_rot1)
    o2, l2 = attend(plan, q_rot2)
    o3, l3 = attend(plan, q_rot1)
    fresh = ForwardPlan(desc, meta)
    o2r, l2r = attend(fresh, q_rot2)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(o1, o3) and torch.equal(l1, l3)
    assert torch.equal(o2, o2r) and torch.equal(l2, l2r)
    assert not torch.equal(o1, o2)
    plan.close()
    fresh.close()
