"""Forward calls on registered working sets (pie_batcher_set_pages /
_submit_forward / _forward_pass) against the Algorithm 2 oracle given the
read/write sets those calls are defined to have: the pages of every slot up to
the call's last row are read, the pages of its new slots written (the sets
Eq. (4) compares, "Pie: Who Should Control the LLM Generation Loop?" §5).  Every
dispatch must agree exactly; every dispatched batch's pass must equal the
folding geometry of "The forward pass" (State geometry) as the Python
marshalling (batching.forward_batch_pass) builds it.  Host code only."""
import random

import numpy as np
import pytest

import oracle.batcher as OB
from programmable_paged_kv_gb300 import Batcher, abi, build
from programmable_paged_kv_gb300.batching import forward_batch_pass


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()


def _sets(pages, first, rows, P):
    """Read and write sets of a forward call at slots [first, first + rows)."""
    last = (first + rows - 1) // P
    return frozenset(int(x) for x in pages[:last + 1]), \
        frozenset(int(x) for x in pages[first // P:last + 1])


@pytest.mark.parametrize("seed", range(24))
def test_forward_calls_match_oracle_and_python_pass(seed):
    rng = random.Random(seed)
    P = rng.choice([8, 16])
    nq = rng.randrange(1, 7)
    nkeys = rng.randrange(1, 6)
    max_calls, max_rows = rng.randrange(1, 9), rng.randrange(4, 60)
    nat = Batcher([True], max_calls, max_rows)
    for _ in range(nq):
        nat.add_queue(0)
    orc = OB.Batcher({q: 0 for q in range(nq)}, {0: True}, max_calls, max_rows)
    # working sets: disjoint page lists, some sharing a prefix page with another
    pool = list(range(400))
    rng.shuffle(pool)
    pages = []
    for k in range(nkeys):
        n = rng.randrange(2, 12)
        own = pool[:n]
        del pool[:n]
        if k and rng.random() < 0.4:
            own = pages[k - 1][:1] + own  # a shared first page
        pages.append(own)
        nat.set_pages(k, own)
    frozen = np.array([rng.randrange(0, 2 * P) for _ in range(nkeys)], np.int32)
    cursor = frozen.astype(np.int64).copy()  # next free slot per key, counting queued calls
    rows_of, key_of = {}, {}
    submitted, in_flight = 0, []
    for _ in range(300):
        act = rng.random()
        if act < 0.35:
            m = rng.randrange(1, 4)
            qs, ks, rs, fs = [], [], [], []
            for _ in range(m):
                q = rng.randrange(nq)
                k = q % nkeys  # a queue works on one working set (queues may share one)
                r = rng.randrange(1, 6)
                if cursor[k] + r > len(pages[k]) * P:
                    continue
                qs.append(q); ks.append(k); rs.append(r); fs.append(int(cursor[k]))
                cursor[k] += r
            if not qs:
                continue
            ids = nat.submit_forward(qs, ks, rs, fs, P)
            assert list(ids) == list(range(submitted, submitted + len(qs)))
            for cid, q, k, r, f in zip(ids, qs, ks, rs, fs):
                rd, wr = _sets(pages[k], f, r, P)
                orc.submit(OB.Call(cid, q, 0, r, (), rd, wr, k))
                rows_of[cid], key_of[cid] = r, k
            submitted += len(qs)
        elif act < 0.55 and in_flight:
            done_ids, lane_keys, rows_per_lane = in_flight.pop(0)  # passes complete in order
            nat.complete(done_ids)
            orc.complete(done_ids)
            for k, n in zip(lane_keys, rows_per_lane):
                frozen[k] += n
        else:
            a = nat.dispatch()
            b = orc.dispatch()
            assert (a is None) == (b is None), (seed, a, b)
            if a is None:
                continue
            assert a == (b.handler, b.calls, b.lane_of_call), (seed, a, b)
            _, ids, lanes = a
            p, lane_keys, first_row = nat.forward_pass(ids, lanes, frozen)
            q_p, q_sets, q_first = forward_batch_pass(ids, lanes, key_of, rows_of, pages,
                                                      [int(x) for x in frozen])
            assert list(lane_keys) == q_sets
            for f in ("row_indptr", "positions", "slots", "kv_len", "page_indptr", "page_ids",
                      "fold_mode"):
                assert np.array_equal(getattr(p, f), getattr(q_p, f)), (seed, f)
            assert [int(x) for x in first_row] == [q_first[c] for c in ids]
            in_flight.append((ids, [int(x) for x in lane_keys],
                              [int(x) for x in np.diff(p.row_indptr)]))


def test_forward_calls_refused():
    b = Batcher([True], 4, 64)
    q = b.add_queue(0)
    with pytest.raises(abi.PieError):
        b.submit_forward([q], [0], [1], [0], 16)  # working set 0 has no pages
    b.set_pages(0, [5, 6])
    with pytest.raises(abi.PieError) as e:
        b.submit_forward([q], [0], [4], [30], 16)  # slots 30..33 past the two pages
    assert e.value.code == abi.PIE_ERANGE
    with pytest.raises(abi.PieError) as e:
        b.set_pages(1, [1 << 26])
    assert e.value.code == abi.PIE_ERANGE
    # a refused submission enqueues nothing
    assert b.counts() == (0, 0)
    ids = b.submit_forward([q, q], [0, 0], [2, 3], [0, 2], 16)
    assert list(ids) == [0, 1]
    _, calls, lanes = b.dispatch()
    assert calls == [0, 1] and lanes == [0, 0]  # one working set: one lane
    p, keys, first = b.forward_pass(calls, lanes, np.array([0], np.int32))
    assert list(p.row_indptr) == [0, 5] and list(p.positions) == [0, 1, 2, 3, 4]
    assert list(p.kv_len) == [5] and list(p.page_ids) == [5, 6] and list(first) == [0, 2]
    with pytest.raises(abi.PieError):
        b.forward_pass(calls, lanes, np.zeros(0, np.int32))  # no frozen length for key 0
