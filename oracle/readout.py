"""Readout distribution epilogue of the oracle: the top-K candidates of a
next-token distribution and their retained mass.

TEST INFRASTRUCTURE ONLY: the test-suite, the package smoke check and the
benchmark's CPU-baseline leg are the only users.  The CUDA library never
imports this module, and this module never imports the library.

Source: the technical review "Pie: Who Should Control the LLM Generation
Loop?", section 7 (sampling access has an information budget), Eq. (6) and
Eq. (7), and the same author's Chinese reading notes, section 7: the serving
system returns, by default, the K = 256 most probable tokens of the
next-token distribution p (a ~128K-token vocabulary) instead of the whole
vector; Z is the probability those tokens keep, q of Eq. (6) is p restricted
to them and divided by Z, and Eq. (7) shows TV(p, q) = 1 - Z.

Readings (where the pages leave a step open):
  * p = softmax(logits) with temperature 1, evaluated here in float64 from
    the logits as given (fp32, or bf16 converted exactly);
  * "the K most probable": sorted by p descending, i.e. by logit
    descending; equal logits are ordered by smaller token id first, so the
    returned ids are unique;
  * the returned probabilities are p itself (not renormalised): the caller
    gets Z and can form q of Eq. (6);
  * lse is the natural-log normaliser log(sum_v exp(logit_v)).
"""
from __future__ import annotations

import numpy as np


def readout_topk(logits: np.ndarray, k: int):
    """logits [R, V] (any float dtype).  Returns (ids int32 [R, k], probs
    float64 [R, k], z float64 [R], lse float64 [R])."""
    x = np.asarray(logits, dtype=np.float64)
    R, V = x.shape
    if not 1 <= k <= V:
        raise ValueError("need 1 <= k <= vocab")
    m = x.max(axis=1)
    lse = m + np.log(np.exp(x - m[:, None]).sum(axis=1))
    ids = np.empty((R, k), np.int32)
    probs = np.empty((R, k), np.float64)
    tok = np.arange(V)
    for r in range(R):
        # lexsort: last key is primary -> logit descending, then id ascending
        order = np.lexsort((tok, -x[r]))[:k]
        ids[r] = order
        probs[r] = np.exp(x[r, order] - lse[r])
    return ids, probs, probs.sum(axis=1), lse


def full_distribution(logits: np.ndarray) -> np.ndarray:
    """p = softmax(logits) per row, float64."""
    x = np.asarray(logits, dtype=np.float64)
    e = np.exp(x - x.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


def renormalised(p: np.ndarray, ids: np.ndarray) -> np.ndarray:
    """q of Eq. (6): p on the returned tokens divided by their mass Z, 0
    elsewhere (one row: p [V], ids [k])."""
    q = np.zeros_like(p)
    z = p[ids].sum()
    q[ids] = p[ids] / z
    return q


def total_variation(p: np.ndarray, q: np.ndarray) -> float:
    """TV(p, q) = 1/2 sum_v |p(v) - q(v)| (the left side of Eq. (7))."""
    return 0.5 * float(np.abs(p - q).sum())
