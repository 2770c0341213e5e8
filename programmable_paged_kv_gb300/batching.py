"""From a dispatched batch of forward calls (Batcher.dispatch) to the
metadata of one multi-lane ForwardPass (pie_fwd_plan): argument marshalling
only.

Every lane of the batch is one working set.  Its calls' rows are
concatenated in batch order and placed at the working set's next free slots
with position = slot (the folding() geometry of "The forward pass", State
geometry); the lane reads kv_len = frozen + rows slots and freezes all of its
new rows.  So a prefix forward and its continuation, merged into one lane by
a vertical group, compute exactly what the two calls compute one after the
other (the continuation's rows see the prefix's rows through slot
causality)."""
from __future__ import annotations

import types

import numpy as np

from .abi import PIE_FOLD_ALL


def forward_batch_pass(call_ids, lanes, call_set, call_rows, set_pages, frozen):
    """call_set[c] / call_rows[c]: the working set and row count of call c;
    set_pages[w]: the physical pages of working set w in slot order;
    frozen[w]: its frozen length before the batch (not modified).
    Returns (pass fields as a namespace, the working set of each lane, the
    first row of each call in the pass)."""
    L = (max(lanes) + 1) if len(lanes) else 0
    lane_set = [None] * L
    lane_rows = [0] * L
    first_row = {}
    for c, l in zip(call_ids, lanes):
        w = call_set[c]
        if lane_set[l] is None:
            lane_set[l] = w
        elif lane_set[l] != w:
            raise ValueError("a lane of the batch spans two working sets")
        lane_rows[l] += call_rows[c]
    if len(set(lane_set)) != L:
        raise ValueError("a working set appears in two lanes of one batch")
    row_indptr = np.zeros(L + 1, np.int32)
    for l in range(L):
        row_indptr[l + 1] = row_indptr[l] + lane_rows[l]
    cursor = row_indptr[:-1].copy()
    for c, l in zip(call_ids, lanes):
        first_row[c] = int(cursor[l])
        cursor[l] += call_rows[c]
    positions = np.concatenate(
        [np.arange(frozen[w], frozen[w] + n, dtype=np.int32) for w, n in zip(lane_set, lane_rows)]
    ) if L else np.zeros(0, np.int32)
    kv_len = np.asarray([frozen[w] + n for w, n in zip(lane_set, lane_rows)], np.int32)
    pages = [np.asarray(set_pages[w], np.int32) for w in lane_set]
    page_indptr = np.zeros(L + 1, np.int32)
    for l in range(L):
        page_indptr[l + 1] = page_indptr[l] + len(pages[l])
    p = types.SimpleNamespace(
        row_indptr=row_indptr, positions=positions, slots=positions.copy(), kv_len=kv_len,
        page_indptr=page_indptr,
        page_ids=np.concatenate(pages) if L else np.zeros(0, np.int32),
        fold_mode=np.full(L, PIE_FOLD_ALL, np.int32), fold_count=np.zeros(L, np.int32),
        mask_word_indptr=None, readout=None)
    return p, lane_set, first_row
