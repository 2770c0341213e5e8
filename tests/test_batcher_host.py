"""The native batcher (pie_batcher_*) against the Algorithm 2 oracle on the
same operation sequences: every dispatch must return the same handler type,
the same call ids in the same order and the same lanes (integer work:
compared exactly).  Plus the calls it refuses.  Host code only: no GPU."""
import ctypes as C
import random

import pytest

import oracle.batcher as OB
from programmable_paged_kv_gb300 import Batcher, abi, build


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()


def _drive(seed, n_calls=120, steps=600):
    rng = random.Random(seed)
    n_types = rng.randrange(1, 4)
    ordered = [rng.random() < 0.6 for _ in range(n_types)]
    nq = rng.randrange(1, 9)
    prios = [rng.randrange(4) for _ in range(nq)]
    max_calls, max_rows = rng.randrange(1, 9), rng.randrange(3, 40)
    nat = Batcher(ordered, max_calls, max_rows)
    for p in prios:
        nat.add_queue(p)
    orc = OB.Batcher({q: p for q, p in enumerate(prios)}, dict(enumerate(ordered)), max_calls,
                     max_rows)
    n_pages = rng.randrange(2, 30)
    submitted, in_flight = 0, []
    for _ in range(steps):
        act = rng.random()
        if act < 0.4 and submitted < n_calls:
            q, h = rng.randrange(nq), rng.randrange(n_types)
            rows = rng.randrange(1, 12)
            deps = sorted({rng.randrange(submitted) for _ in range(rng.randrange(3))}) if submitted else []
            reads = [rng.randrange(n_pages) for _ in range(rng.randrange(4))]
            writes = [rng.randrange(n_pages) for _ in range(rng.randrange(3))]
            key = rng.randrange(-1, 4)
            cid = nat.submit(q, h, rows, key, deps, reads, writes)
            assert cid == submitted
            orc.submit(OB.Call(cid, q, h, rows, tuple(deps), frozenset(reads), frozenset(writes),
                               key))
            submitted += 1
        elif act < 0.6 and in_flight:
            done = in_flight.pop(rng.randrange(len(in_flight)))
            nat.complete(done)
            orc.complete(done)
        else:
            a = nat.dispatch()
            b = orc.dispatch()
            assert (a is None) == (b is None), (seed, a, b)
            if a is not None:
                assert a == (b.handler, b.calls, b.lane_of_call), (seed, a, b)
                in_flight.append(a[1])
    queued, flying = nat.counts()
    assert flying == sum(len(x) for x in in_flight)
    assert queued == sum(len(v) for v in orc.pending.values())
    nat.close()


@pytest.mark.parametrize("seed", range(60))
def test_native_batcher_matches_the_oracle(seed):
    _drive(seed)


def test_native_batcher_large_trace():
    # many queues and calls: the same decisions at scale
    _drive(1234, n_calls=3000, steps=12000)


def test_batcher_refusals():
    lib = abi.load()
    h = C.c_void_p()
    assert lib.pie_batcher_create(0, None, 4, 16, C.byref(h)) == abi.PIE_EINVAL
    assert lib.pie_batcher_create(2, None, 0, 16, C.byref(h)) == abi.PIE_EINVAL
    assert lib.pie_batcher_create(2, None, 4, 0, C.byref(h)) == abi.PIE_EINVAL
    b = Batcher([True, False], 4, 16)
    q = b.add_queue(1)
    cid = C.c_int64()
    sub = lambda *a: lib.pie_batcher_submit(b.handle, *a, C.byref(cid))
    assert sub(5, 0, 1, -1, None, 0, None, 0, None, 0) == abi.PIE_EINVAL     # unknown queue
    assert sub(q, 2, 1, -1, None, 0, None, 0, None, 0) == abi.PIE_EINVAL     # unknown handler
    assert sub(q, 0, 0, -1, None, 0, None, 0, None, 0) == abi.PIE_EINVAL     # rows < 1
    dep = (C.c_int64 * 1)(0)
    assert sub(q, 0, 1, -1, dep, 1, None, 0, None, 0) == abi.PIE_EINVAL      # not an earlier call
    assert sub(q, 0, 1, -1, None, 1, None, 0, None, 0) == abi.PIE_EINVAL     # NULL with a count
    big = (C.c_int64 * 1)(1 << 26)
    neg = (C.c_int64 * 1)(-1)
    assert sub(q, 0, 1, -1, None, 0, big, 1, None, 0) == abi.PIE_ERANGE      # resource id too large
    assert sub(q, 0, 1, -1, None, 0, None, 0, neg, 1) == abi.PIE_ERANGE      # negative resource id
    assert b.submit(q, 0, 1) == 0
    n, hh = C.c_int32(), C.c_int32()
    small = (C.c_int64 * 2)()
    lanes = (C.c_int32 * 2)()
    assert lib.pie_batcher_dispatch(b.handle, small, lanes, 2, C.byref(n), C.byref(hh)) == abi.PIE_ENOSPACE
    assert b.counts() == (1, 0)
    assert lib.pie_batcher_complete(b.handle, (C.c_int64 * 1)(0), 1) == abi.PIE_EINVAL  # still queued
    assert b.dispatch() == (0, [0], [0])
    assert b.counts() == (0, 1)
    b.complete([0])
    assert b.counts() == (0, 0)
    assert lib.pie_batcher_complete(b.handle, (C.c_int64 * 1)(0), 1) == abi.PIE_EINVAL  # twice
    assert b.dispatch() is None
    b.close()


@pytest.mark.parametrize("seed", range(12))
def test_submit_many_matches_one_by_one(seed):
    # the same operations, calls submitted one by one into one batcher and in
    # random groups into the other: the same ids and the same batches
    rng = random.Random(seed)
    nq = rng.randrange(1, 7)
    ordered = [rng.random() < 0.6 for _ in range(2)]
    a, b = Batcher(ordered, 6, 24), Batcher(ordered, 6, 24)
    prios = [rng.randrange(3) for _ in range(nq)]
    for p in prios:
        a.add_queue(p)
        b.add_queue(p)
    submitted, flying = 0, []
    for _ in range(300):
        act = rng.random()
        if act < 0.45 and submitted < 200:
            group = []
            for _ in range(rng.randrange(1, 6)):
                cid = submitted + len(group)
                deps = sorted({rng.randrange(cid) for _ in range(rng.randrange(3))}) if cid else []
                group.append((rng.randrange(nq), rng.randrange(2), rng.randrange(1, 6),
                              rng.randrange(-1, 3), deps,
                              [rng.randrange(20) for _ in range(rng.randrange(4))],
                              [rng.randrange(20) for _ in range(rng.randrange(2))]))
            for g in group:
                assert a.submit(g[0], g[1], g[2], g[3], g[4], g[5], g[6]) == submitted
                submitted += 1
            ids = b.submit_many(*[[g[f] for g in group] for f in range(7)])
            assert list(ids) == list(range(submitted - len(group), submitted))
        elif act < 0.65 and flying:
            done = flying.pop(rng.randrange(len(flying)))
            a.complete(done)
            b.complete(done)
        else:
            x, y = a.dispatch(), b.dispatch()
            assert x == y, (seed, x, y)
            if x is not None:
                flying.append(x[1])
        assert a.counts() == b.counts()
    a.close()
    b.close()


def test_submit_many_refusals_change_nothing():
    b = Batcher([True], 4, 16)
    q = b.add_queue(0)
    assert list(b.submit_many([q], [0], [1], [-1], [[]], [[1]], [[2]])) == [0]
    # the third call names a dependency that is not earlier: nothing is enqueued
    with pytest.raises(Exception):
        b.submit_many([q, q, q], [0, 0, 0], [1, 1, 1], [-1, -1, -1], [[0], [1], [5]],
                      [[], [], []], [[], [], []])
    assert b.counts() == (1, 0)
    # a resource id out of range in the last call: nothing is enqueued
    with pytest.raises(Exception):
        b.submit_many([q, q], [0, 0], [1, 1], [-1, -1], [[], []], [[3], [1 << 26]], [[], []])
    assert b.counts() == (1, 0)
    # the ids continue where they were
    assert list(b.submit_many([q, q], [0, 0], [1, 1], [-1, -1], [[], [1]], [[], []],
                              [[], []])) == [1, 2]
    assert list(b.submit_many([], [], [], [], [], [], [])) == []
    assert b.counts() == (3, 0)
    b.close()
