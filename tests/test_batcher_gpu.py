"""Forward calls of many command queues through the work-conserving batcher
(pie_batcher_*) and the ForwardPass (pie_fwd_*): one multi-lane pass per
dispatched batch, vertical groups merged into one lane.  Every call's
outputs and the final pools must equal the oracle running each call alone,
queue by queue: batching across queues and within a queue preserves meaning
(the Pie review, section 5; the prefix-and-continuation case of Fig. 4)."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests.parity import assert_bits_equal, assert_lse_close, assert_out_close, assert_rope_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from programmable_paged_kv_gb300 import build
    build()


def submit_trace(trace, batcher, native=False):
    """Queue every call of the trace; its reads are the pages it attends over,
    its writes the pages of its new slots (native: the batcher derives both
    from the queue's registered working set).  Returns the call tables."""
    P = trace.pool.desc.page_size
    qids = [batcher.add_queue(int(p)) for p in trace.priority]
    cursor = [int(c) for c in trace.cached]
    call_set, call_rows, call_inputs = {}, {}, {}
    if native:
        for q, pages in enumerate(trace.queue_pages):
            batcher.set_pages(q, pages)
    for q, qq, kk, vv in trace.calls:
        n = qq.shape[0]
        pages = trace.queue_pages[q]
        writes = sorted({int(pages[s // P]) for s in range(cursor[q], cursor[q] + n)})
        reads = [int(x) for x in pages[:(cursor[q] + n + P - 1) // P]]
        if native:
            cid = batcher.submit_forward([qids[q]], [q], [n], [cursor[q]], P)[0]
        else:
            cid = batcher.submit(qids[q], 0, n, key=q, reads=reads, writes=writes)
        cursor[q] += n
        call_set[cid], call_rows[cid], call_inputs[cid] = q, n, (qq, kk, vv)
    return call_set, call_rows, call_inputs


def run_batched(trace, max_calls, max_rows, native=False):
    import torch
    from programmable_paged_kv_gb300 import Batcher, ForwardPlan, make_desc, make_meta, runner
    from programmable_paged_kv_gb300.batching import forward_batch_pass
    d = trace.pool.desc
    desc = make_desc(d)
    pools = runner.DevicePools(trace.pool)
    b = Batcher([True], max_calls, max_rows)
    call_set, call_rows, call_inputs = submit_trace(trace, b, native)
    frozen = {q: int(c) for q, c in enumerate(trace.cached)}
    frozen_arr = np.asarray(trace.cached, np.int32).copy()
    tdt = torch.bfloat16 if d.dtype == W.BF16 else torch.float32
    Hq, Hkv, D = d.num_q_heads, d.num_kv_heads, d.head_dim
    outs, batches = {}, []
    while True:
        r = b.dispatch()
        if r is None:
            break
        _, ids, lanes = r
        if native:
            # built and planned in one native call
            ws = torch.empty(1 << 22, dtype=torch.uint8, device="cuda")
            plan, keys, first_arr, kv_len, N = b.plan_forward(ids, lanes, frozen_arr, desc,
                                                              trace.pool.num_pool_pages, ws)
            lane_set = [int(x) for x in keys]
            first = {c: int(f) for c, f in zip(ids, first_arr)}
            kv_len = kv_len.copy()
            rows_of = [int(x) - frozen[w] for x, w in zip(kv_len, lane_set)]
        else:
            p, lane_set, first = forward_batch_pass(ids, lanes, call_set, call_rows,
                                                    trace.queue_pages, frozen)
            N = int(p.row_indptr[-1])
            plan = ForwardPlan(desc, make_meta(p, trace.pool.num_pool_pages))
            kv_len, rows_of = p.kv_len, np.diff(p.row_indptr)
        q = np.empty((N, Hq, D), trace.calls[0][1].dtype)
        k = np.empty((N, Hkv, D), q.dtype)
        v = np.empty((N, Hkv, D), q.dtype)
        for c in ids:
            s = slice(first[c], first[c] + call_rows[c])
            q[s], k[s], v[s] = call_inputs[c]
        fr = torch.tensor([frozen[w] for w in lane_set], dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        q_rot = torch.empty((N, Hq, D), dtype=tdt, device="cuda")
        plan.append_kv(runner.to_device(q, d.dtype), runner.to_device(k, d.dtype),
                       runner.to_device(v, d.dtype), q_rot, pools.k, pools.v, fr, st)
        out = torch.empty((N, Hq, D), dtype=tdt, device="cuda")
        lse = torch.empty((N, Hq), dtype=torch.float32, device="cuda")
        plan.attend(q_rot, pools.k, pools.v, None, None, None, out, lse, st)
        plan.fold(fr, None, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert np.array_equal(fr.cpu().numpy(), kv_len), "fold must freeze every new row"
        out_h, lse_h = runner.to_host(out, d.dtype), lse.cpu().numpy()
        for c in ids:
            s = slice(first[c], first[c] + call_rows[c])
            outs[c] = (out_h[s], lse_h[s])
        for w, n in zip(lane_set, rows_of):
            frozen[w] += int(n)
            frozen_arr[w] += int(n)
        plan.close()
        b.complete(ids)
        batches.append((ids, lanes))
    assert b.counts() == (0, 0)
    b.close()
    k_used = runner.to_host(pools.k.index_select(0, pools.used), d.dtype)
    v_used = runner.to_host(pools.v.index_select(0, pools.used), d.dtype)
    return outs, k_used, v_used, batches, runner._untouched_is_canary(pools, d.dtype)


def run_alone(trace):
    """The oracle: each call as its own one-lane pass, in arrival order (queue
    order within each queue; queues share only frozen, read-only pages)."""
    sc = trace.pool
    k, v = sc.k_init.copy(), sc.v_init.copy()
    frozen = [int(c) for c in trace.cached]
    outs = {}
    for cid, (q, qq, kk, vv) in enumerate(trace.calls):
        n = qq.shape[0]
        pages = trace.queue_pages[q]
        pos = np.arange(frozen[q], frozen[q] + n, dtype=np.int32)
        p = W.Pass(row_indptr=np.array([0, n], np.int32), positions=pos, slots=pos.copy(),
                   kv_len=np.array([frozen[q] + n], np.int32),
                   page_indptr=np.array([0, len(pages)], np.int32), page_ids=pages,
                   fold_mode=np.array([1], np.int32), fold_count=np.zeros(1, np.int32),
                   q=qq, k=kk, v=vv)
        fr = np.array([frozen[q]], np.int32)
        r = O.run_pass(sc.desc, p, k, v, fr, page_ids=sc.compact_page_ids(pages))
        assert r["err"] == O.OK
        assert r["status"] == 0
        frozen[q] = int(fr[0])
        outs[cid] = (r["out"], r["lse"])
    return outs, k, v


@pytest.mark.parametrize("limits,native", [((16, 512), False), ((4, 64), False), ((1, 1), False),
                                           ((16, 512), True), ((4, 64), True)],
                         ids=["wide", "narrow", "one_call", "wide_native", "narrow_native"])
def test_batched_calls_equal_calls_run_alone(limits, native):
    trace = W.forward_calls(3, queues=12, calls_per_queue=5, prefix=64, private_hi=40,
                            prefill_lo=4, prefill_hi=40, desc=W.Desc(8, 2, 128, 16, W.BF16),
                            num_pool_pages=1024)
    outs, k_used, v_used, batches, untouched = run_batched(trace, *limits, native)
    ref, k_ref, v_ref = run_alone(trace)
    dt = trace.pool.desc.dtype
    assert untouched
    assert sorted(outs) == list(range(len(trace.calls)))
    for c in range(len(trace.calls)):
        assert_out_close(outs[c][0], ref[c][0], dt, f"call {c} out")
        assert_lse_close(outs[c][1], ref[c][1], dt, f"call {c} lse")
    assert_rope_close(k_used, k_ref, dt, "K pool")
    assert_bits_equal(v_used, v_ref, "V pool")
    if limits[0] > 1:
        # the trace exercised both kinds of batching
        assert any(len(set(l)) > 1 for _, l in batches), "no batch held two lanes"
        assert any(len(l) > len(set(l)) for _, l in batches), "no lane merged two calls"
    else:
        assert all(len(ids) == 1 for ids, _ in batches)
