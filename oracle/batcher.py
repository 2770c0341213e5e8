"""Work-conserving dispatch of API calls (Algorithm 2), in the oracle.

TEST INFRASTRUCTURE ONLY: the test-suite and the benchmark's CPU-baseline
leg are the only users.  The native batcher never imports this module, and
this module never imports the library.

Source: the Pie review, section 5 ("Batching API calls while preserving
meaning"), Algorithm 2 ("Work-conserving API dispatch") and Eq. (4), with the
paper's horizontal and vertical batching (Fig. 4).  GPU-bound calls wait in
their command queues in arrival order; whenever the GPU is idle the
controller forms one batch: eligible calls per handler type, compatible calls
combined across queues, vertical groups within a queue, ordered by queue
priority, truncated at the backend limit; the candidate holding the oldest
pending call is dispatched; completions make dependents eligible.

Readings (the page leaves these steps abstract):
  * calls carry an arrival id (0, 1, 2, ... = age), a queue, a handler type,
    a row count, explicit dependencies (ids of earlier calls), the resources
    they read and write (e.g. KV pages) and a working-set key;
  * queue order is kept: a queue contributes only through its oldest pending
    call, and only once every dependency of that call has completed;
  * a vertical group is that head plus the following pending calls of the same
    queue and handler type, in order, while each one's dependencies are
    completed or earlier in the group; only handler types that keep order
    inside a batch (a forward pass does: its scatter runs before its
    attention) form groups longer than one call;
  * groups of one handler type are taken in queue-priority order (higher
    first, then the group holding the older call); a group joins the
    candidate only if Eq. (4) holds between its resources and those of every
    group already taken (a group's own calls may touch the same resources:
    their order is kept inside the batch);
  * truncation walks the ordered calls and stops at the first call that
    would exceed max_calls or max_rows; a batch always keeps its first call;
  * among handler types the candidate whose smallest call id is smallest is
    dispatched;
  * consecutive calls of one group with the same working-set key become one
    lane of the pass (a prefix forward and its continuation); every other
    call is a lane of its own.
Algorithm 2 is a policy, so there is no closed form to test it against: the
pins check it against hand-worked traces and against the properties the
pages state (queue order, dependencies, Eq. (4), limits, work conservation,
oldest-call choice).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, FrozenSet, List, Optional, Tuple


@dataclasses.dataclass(frozen=True)
class Call:
    id: int
    queue: int
    handler: int
    rows: int
    deps: Tuple[int, ...] = ()
    reads: FrozenSet[int] = frozenset()
    writes: FrozenSet[int] = frozenset()
    key: int = -1


@dataclasses.dataclass
class Batch:
    handler: int
    calls: List[int]        # call ids in dispatch order
    lane_of_call: List[int]  # lane index of each call (same length)


def independent(r_a, w_a, r_b, w_b) -> bool:
    """Eq. (4): W(a) does not meet R(b) | W(b), and W(b) does not meet R(a) | W(a)."""
    return not (w_a & (r_b | w_b)) and not (w_b & (r_a | w_a))


class Batcher:
    def __init__(self, priorities: Dict[int, int], vertical: Dict[int, bool],
                 max_calls: int, max_rows: int):
        self.priorities = dict(priorities)
        self.vertical = dict(vertical)
        self.max_calls = max_calls
        self.max_rows = max_rows
        self.calls: Dict[int, Call] = {}
        self.pending: Dict[int, List[int]] = {q: [] for q in priorities}  # queue -> ids, in order
        self.done: set = set()

    # arrival (Algorithm 2): identify the queue and dependencies, enqueue in order
    def submit(self, call: Call):
        assert call.id not in self.calls
        for d in call.deps:
            assert d < call.id
        self.calls[call.id] = call
        self.pending[call.queue].append(call.id)

    # completion (Algorithm 2): completions make dependents eligible
    def complete(self, ids):
        self.done.update(ids)

    def _group(self, q: int) -> List[int]:
        """Line 06/08: the queue's eligible head and its vertical group."""
        ids = self.pending[q]
        if not ids:
            return []
        head = self.calls[ids[0]]
        if not all(d in self.done for d in head.deps):
            return []
        group = [head.id]
        if not self.vertical.get(head.handler, False):
            return group
        for cid in ids[1:]:
            c = self.calls[cid]
            if c.handler != head.handler:
                break
            if not all(d in self.done or d in group for d in c.deps):
                break
            group.append(cid)
        return group

    def _candidate(self, handler: int, groups: List[List[int]]) -> List[Tuple[int, List[int]]]:
        """Lines 07, 09, 10 for one handler type: combine groups across queues in
        priority order under Eq. (4), then truncate at the limits."""
        order = sorted(groups, key=lambda g: (-self.priorities[self.calls[g[0]].queue], g[0]))
        taken: List[List[int]] = []
        res: List[Tuple[FrozenSet[int], FrozenSet[int]]] = []
        for g in order:
            r = frozenset().union(*(self.calls[c].reads for c in g))
            w = frozenset().union(*(self.calls[c].writes for c in g))
            if all(independent(r, w, r2, w2) for r2, w2 in res):
                taken.append(g)
                res.append((r, w))
        out: List[Tuple[int, List[int]]] = []
        n_calls = n_rows = 0
        stop = False
        for gi, g in enumerate(taken):
            kept = []
            for c in g:
                rows = self.calls[c].rows
                if n_calls > 0 and (n_calls + 1 > self.max_calls or n_rows + rows > self.max_rows):
                    stop = True
                    break
                kept.append(c)
                n_calls += 1
                n_rows += rows
            if kept:
                out.append((gi, kept))
            if stop:
                break
        return out

    # GPU idle (Algorithm 2): one dispatch
    def dispatch(self) -> Optional[Batch]:
        by_handler: Dict[int, List[List[int]]] = {}
        for q in self.pending:
            g = self._group(q)
            if g:
                by_handler.setdefault(self.calls[g[0]].handler, []).append(g)
        best = None
        for h, groups in by_handler.items():
            cand = self._candidate(h, groups)
            oldest = min(c for _, kept in cand for c in kept)
            if best is None or oldest < best[0]:
                best = (oldest, h, cand)
        if best is None:
            return None
        _, h, cand = best
        calls, lanes = [], []
        lane = -1
        for _, kept in cand:
            prev_key = None
            for i, c in enumerate(kept):
                key = self.calls[c].key
                if i == 0 or key < 0 or key != prev_key:
                    lane += 1
                prev_key = key
                calls.append(c)
                lanes.append(lane)
        for c in calls:
            self.pending[self.calls[c].queue].remove(c)
        return Batch(h, calls, lanes)


def run_trace(priorities, vertical, max_calls, max_rows, arrivals, service):
    """Drive the batcher as the control layer would: `arrivals` is a list of
    (time, Call) sorted by time; a dispatched batch occupies the GPU for
    service(batch) time units and completes at its end; the GPU dispatches
    whenever it is idle and a batch can be formed (work conservation).
    Returns [(dispatch time, Batch)]."""
    b = Batcher(priorities, vertical, max_calls, max_rows)
    t, i, out = 0.0, 0, []
    busy_until, in_flight = 0.0, None
    n = len(arrivals)
    while i < n or in_flight is not None or any(b.pending[q] for q in b.pending):
        # completion of the batch in flight
        if in_flight is not None and t >= busy_until:
            b.complete(in_flight.calls)
            in_flight = None
        while i < n and arrivals[i][0] <= t:
            b.submit(arrivals[i][1])
            i += 1
        if in_flight is None:
            batch = b.dispatch()
            if batch is not None:
                out.append((t, batch))
                in_flight = batch
                busy_until = t + service(batch)
                continue
        # advance to the next event
        nxt = []
        if in_flight is not None:
            nxt.append(busy_until)
        if i < n:
            nxt.append(arrivals[i][0])
        if not nxt:
            break  # calls left whose dependencies can never complete
        t = max(t, min(nxt))
    return out
