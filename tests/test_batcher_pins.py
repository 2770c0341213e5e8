"""Pins of the Algorithm 2 oracle (Pie review, section 5: work-conserving API
dispatch, Eq. (4), horizontal and vertical batching) against hand-worked
traces and the properties the pages state: queue order kept, dependencies
honoured, Eq. (4) between queues of one batch, backend limits, work
conservation, the oldest-call choice between handler types.  Mistakes planted
in copies of the oracle must each fail a pin."""
import random
import sys
import types

import pytest

import oracle.batcher as OB

FWD, EMBED = 0, 1
VERT = {FWD: True, EMBED: False}


def C(i, q, h, rows, deps=(), reads=(), writes=(), key=-1):
    return OB.Call(i, q, h, rows, tuple(deps), frozenset(reads), frozenset(writes), key)


def _batches(ob, prios, calls, max_calls=8, max_rows=100, script=()):
    """Submit `calls`, then run `script`: 'd' = dispatch (recorded), ('c', ids) =
    complete.  Returns the recorded dispatches as (handler, calls, lanes)."""
    b = ob.Batcher(prios, VERT, max_calls, max_rows)
    for c in calls:
        b.submit(c)
    out = []
    for step in script:
        if step == "d":
            r = b.dispatch()
            out.append(None if r is None else (r.handler, r.calls, r.lane_of_call))
        else:
            b.complete(step[1])
    return out


def pin_hand_horizontal_vertical(ob):
    # a prefix forward and its continuation (vertical group, one lane); a
    # forward of another queue that reads the prefix's page (Eq. (4) conflict,
    # left for later); an embedding in a higher-priority queue ahead of a forward
    calls = [C(0, 0, FWD, 4, writes={10}, key=100),
             C(1, 1, EMBED, 1),
             C(2, 1, FWD, 2, writes={20}, key=200),
             C(3, 2, FWD, 3, reads={10}, writes={30}, key=300),
             C(4, 0, FWD, 1, deps=(0,), reads={10}, writes={10}, key=100)]
    got = _batches(ob, {0: 1, 1: 2, 2: 1}, calls, script=["d", "d", "d", "d"])
    assert got == [(FWD, [0, 4], [0, 0]), (EMBED, [1], [0]), (FWD, [2, 3], [0, 1]), None]


def pin_hand_priority_truncation(ob):
    # the backend takes 3 calls / 10 rows; priority decides who is cut, even the oldest call
    calls = [C(0, 0, FWD, 4, key=0), C(1, 1, FWD, 5, key=1), C(2, 2, FWD, 3, key=2),
             C(3, 3, FWD, 1, key=3), C(4, 1, FWD, 1, key=4)]
    got = _batches(ob, {0: 1, 1: 3, 2: 2, 3: 1}, calls, max_calls=3, max_rows=10,
                   script=["d", "d", "d"])
    assert got == [(FWD, [1, 4, 2], [0, 1, 2]), (FWD, [0, 3], [0, 1]), None]
    # rows, not calls, bind: 5 + 1 + 3 = 9 <= 10, a fourth call would make 13
    got = _batches(ob, {0: 1, 1: 3, 2: 2, 3: 1}, calls, max_calls=8, max_rows=10,
                   script=["d", "d"])
    assert got == [(FWD, [1, 4, 2], [0, 1, 2]), (FWD, [0, 3], [0, 1])]
    # a call larger than the row limit still goes, alone
    got = _batches(ob, {0: 1}, [C(0, 0, FWD, 50), C(1, 0, EMBED, 1)], max_rows=10,
                   script=["d", "d"])
    assert got == [(FWD, [0], [0]), (EMBED, [1], [0])]


def pin_hand_oldest_between_types(ob):
    # priority orders calls inside a batch; between handler types the oldest call wins
    calls = [C(0, 0, EMBED, 1), C(1, 1, FWD, 1, key=1), C(2, 2, EMBED, 1)]
    got = _batches(ob, {0: 1, 1: 5, 2: 9}, calls, script=["d", "d", "d"])
    assert got == [(EMBED, [2, 0], [0, 1]), (FWD, [1], [0]), None]
    # the oldest call is judged inside each truncated candidate: embeddings cut to
    # the high-priority queue's call (id 3) lose to a forward holding id 1
    calls = [C(0, 0, EMBED, 1), C(1, 1, FWD, 1, key=1), C(2, 2, FWD, 1, key=2),
             C(3, 3, EMBED, 1)]
    got = _batches(ob, {0: 1, 1: 1, 2: 1, 3: 9}, calls, max_calls=1, script=["d", "d", "d", "d"])
    assert got == [(FWD, [1], [0]), (FWD, [2], [0]), (EMBED, [3], [0]), (EMBED, [0], [0])]


def pin_hand_dependencies(ob):
    # a call waits for its dependency's completion; a vertical group stops at a
    # call that depends on another queue's unfinished work
    calls = [C(0, 0, FWD, 1, key=0), C(1, 1, FWD, 1, deps=(0,), key=1),
             C(2, 0, FWD, 1, deps=(1,), key=0), C(3, 0, FWD, 1, deps=(0,), key=0)]
    got = _batches(ob, {0: 1, 1: 1}, calls,
                   script=["d", "d", ("c", [0]), "d", "d", ("c", [1]), "d", "d"])
    assert got == [(FWD, [0], [0]), None, (FWD, [1], [0]), None, (FWD, [2, 3], [0, 0]), None]
    # embeddings never form vertical groups
    got = _batches(ob, {0: 1}, [C(0, 0, EMBED, 1), C(1, 0, EMBED, 1)], script=["d", "d"])
    assert got == [(EMBED, [0], [0]), (EMBED, [1], [0])]
    # a vertical group ends at the first call of another type
    calls = [C(0, 0, FWD, 1, key=7), C(1, 0, EMBED, 1), C(2, 0, FWD, 1, key=7)]
    got = _batches(ob, {0: 1}, calls, script=["d", "d", "d"])
    assert got == [(FWD, [0], [0]), (EMBED, [1], [0]), (FWD, [2], [0])]
    # one group, two working sets: two lanes
    calls = [C(0, 0, FWD, 1, key=7), C(1, 0, FWD, 1, key=8), C(2, 0, FWD, 1, key=8)]
    got = _batches(ob, {0: 1}, calls, script=["d"])
    assert got == [(FWD, [0, 1, 2], [0, 1, 1])]


def _random_calls(rng, n, nq):
    calls = []
    for i in range(n):
        q = rng.randrange(nq)
        h = FWD if rng.random() < 0.7 else EMBED
        deps = []
        if i and rng.random() < 0.3:
            deps.append(rng.randrange(i))
        pages = list(range(12))
        reads = set(rng.sample(pages, rng.randrange(3)))
        writes = set(rng.sample(pages, rng.randrange(2)))
        calls.append(C(i, q, h, rng.randrange(1, 9), deps, reads, writes, key=rng.randrange(3)))
    return calls


def pin_properties_on_random_traces(ob):
    """Queue order, dependencies, Eq. (4), limits and work conservation after
    every dispatch of random traces (checked directly, not through the oracle)."""
    for seed in range(40):
        rng = random.Random(seed)
        nq = rng.randrange(1, 6)
        prios = {q: rng.randrange(4) for q in range(nq)}
        max_calls, max_rows = rng.randrange(1, 7), rng.randrange(4, 20)
        b = ob.Batcher(prios, VERT, max_calls, max_rows)
        calls = _random_calls(rng, 30, nq)
        byid = {c.id: c for c in calls}
        dispatched, completed, in_flight = [], set(), []
        for c in calls[:10]:
            b.submit(c)
        nxt = 10
        for _ in range(200):
            act = rng.random()
            if act < 0.3 and nxt < len(calls):
                b.submit(calls[nxt])
                nxt += 1
                continue
            if act < 0.55 and in_flight:
                done = in_flight.pop(0)
                b.complete(done)
                completed.update(done)
                continue
            r = b.dispatch()
            submitted = [c for c in calls[:nxt]]
            if r is None:
                # work conservation: no queue head is ready
                for q in range(nq):
                    pend = [c for c in submitted if c.queue == q and c.id not in dispatched]
                    if pend:
                        assert not all(d in completed for d in pend[0].deps)
                continue
            ids = r.calls
            assert ids and len(ids) == len(r.lane_of_call)
            assert len({byid[i].handler for i in ids}) == 1 and byid[ids[0]].handler == r.handler
            assert len(ids) <= max_calls or len(ids) == 1
            assert len(ids) == 1 or sum(byid[i].rows for i in ids) <= max_rows
            for k, i in enumerate(ids):
                c = byid[i]
                # queue order: every earlier call of the queue went before or earlier here
                for e in submitted:
                    if e.queue == c.queue and e.id < c.id:
                        assert e.id in dispatched or e.id in ids[:k]
                # dependencies: completed, or earlier in this batch and in the same queue
                for d in c.deps:
                    assert d in completed or (d in ids[:k] and byid[d].queue == c.queue)
            for i in ids:
                for j in ids:
                    a, bb = byid[i], byid[j]
                    if a.queue != bb.queue:
                        assert OB.independent(a.reads, a.writes, bb.reads, bb.writes)
            # lanes: consecutive, a new lane unless same queue and same key as the previous call
            for k in range(1, len(ids)):
                a, bb = byid[ids[k - 1]], byid[ids[k]]
                same = a.queue == bb.queue and a.key == bb.key and a.key >= 0
                assert r.lane_of_call[k] == r.lane_of_call[k - 1] + (0 if same else 1)
            dispatched.extend(ids)
            in_flight.append(list(ids))


def pin_trace_is_work_conserving(ob):
    # the GPU never idles while a batch can be formed: a batch starts at every
    # completion or arrival instant that finds the GPU idle
    arrivals = [(0.0, C(0, 0, FWD, 2, key=0)), (0.5, C(1, 1, FWD, 2, key=1)),
                (0.6, C(2, 2, EMBED, 1)), (5.0, C(3, 0, FWD, 1, deps=(0,), key=0))]
    out = ob.run_trace({0: 1, 1: 1, 2: 1}, VERT, 8, 100, arrivals, lambda b: 1.0)
    got = [(t, b.handler, b.calls) for t, b in out]
    assert got == [(0.0, FWD, [0]), (1.0, FWD, [1]), (2.0, EMBED, [2]), (5.0, FWD, [3])]


PINS = [pin_hand_horizontal_vertical, pin_hand_priority_truncation, pin_hand_oldest_between_types,
        pin_hand_dependencies, pin_properties_on_random_traces, pin_trace_is_work_conserving]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_batcher_oracle_pins(pin):
    pin(OB)


MUTANTS = {
    "priority_reversed": ("key=lambda g: (-self.priorities[", "key=lambda g: (self.priorities["),
    "no_eq4_check": ("if all(independent(r, w, r2, w2) for r2, w2 in res):", "if True:"),
    "head_deps_ignored": ("if not all(d in self.done for d in head.deps):\n            return []",
                          "if False:\n            return []"),
    "youngest_wins": ("if best is None or oldest < best[0]:", "if best is None or oldest > best[0]:"),
    "vertical_mixes_types": ("            if c.handler != head.handler:\n                break\n", ""),
    "truncation_skips": ("                    stop = True\n                    break", "                    continue"),
    "lanes_never_merge": ("if i == 0 or key < 0 or key != prev_key:", "if True:"),
    "group_dep_outside": ("if not all(d in self.done or d in group for d in c.deps):",
                          "if not all(d in self.done or d in self.calls for d in c.deps):"),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_mistakes_fail_a_pin(name):
    src = open(OB.__file__).read()
    a, b = MUTANTS[name]
    assert src.count(a) == 1, name
    mod = types.ModuleType("batcher_mutant")
    sys.modules["batcher_mutant"] = mod  # dataclasses look their module up
    try:
        exec(compile(src.replace(a, b), "batcher_mutant", "exec"), mod.__dict__)
    finally:
        sys.modules.pop("batcher_mutant", None)
    failed = 0
    for pin in PINS:
        try:
            pin(mod)
        except (AssertionError, ValueError, KeyError, IndexError):
            failed += 1
    assert failed > 0, f"mutant {name} passed every pin"
