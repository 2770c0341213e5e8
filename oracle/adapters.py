"""Per-lane adapters at a projection site, in the oracle.

TEST INFRASTRUCTURE ONLY: the test-suite, the package smoke check and the
benchmark's CPU-baseline leg are the only users.  The CUDA library never
imports this module, and this module never imports the library.

Source: Pie documentation, "The forward pass", section Adapters: an adapter
attached at a projection site ("q", "k", "v", "o", "gate_up", "down") is a
function f(x, y) of the projection input x and its base output y that returns
the output; the one interface covers LoRA (y + b (a x)) and IA3 (y scaled),
and concurrent requests in one batch may use different adapters.

Readings (where the page leaves a step open):
  * an adapter a holds a LoRA pair A_a [r][d_in], B_a [d_out][r] with a
    scalar scale_a (the usual alpha / r; 0 turns LoRA off) and an IA3
    vector s_a [d_out] (all ones when the adapter has no IA3 part); applied
    to a row as  y' = (y + scale_a * B_a (A_a x)) * s_a  (elementwise in s_a);
  * every row of a lane uses the lane's adapter; a lane with adapter -1 keeps
    y unchanged;
  * x, y, A, B and s are of the pass dtype; the oracle computes in float64
    and rounds y' to the dtype once.
DoRA (also named on the page) needs the base weight's column norms, which a
projection site's (x, y) do not carry: it is not built.
"""
from __future__ import annotations

from typing import Optional

import numpy as np


def apply_adapters(x: np.ndarray, y: np.ndarray, row_indptr: np.ndarray,
                   adapter_of_lane: np.ndarray, A: np.ndarray, B: np.ndarray,
                   scale: np.ndarray, ia3: Optional[np.ndarray]) -> np.ndarray:
    """x [N, d_in], y [N, d_out] (float arrays holding the dtype's values),
    row_indptr [L+1], adapter_of_lane [L] (-1: none), A [n_ad, r, d_in],
    B [n_ad, d_out, r], scale [n_ad], ia3 [n_ad, d_out] or None.
    Returns y' [N, d_out] in float64 (before rounding to the dtype)."""
    x = np.asarray(x, np.float64)
    out = np.asarray(y, np.float64).copy()
    for l in range(len(adapter_of_lane)):
        a = int(adapter_of_lane[l])
        r0, r1 = int(row_indptr[l]), int(row_indptr[l + 1])
        if a < 0 or r1 == r0:
            continue
        t = x[r0:r1] @ np.asarray(A[a], np.float64).T          # [n, r]
        yl = out[r0:r1] + float(scale[a]) * (t @ np.asarray(B[a], np.float64).T)
        if ia3 is not None:
            yl = yl * np.asarray(ia3[a], np.float64)[None, :]
        out[r0:r1] = yl
    return out
