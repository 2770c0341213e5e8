"""Pins of the readout oracle (top-K of the next-token distribution, the
review "Pie: Who Should Control the LLM Generation Loop?", section 7,
Eq. (6)-(7)) against facts fixed outside it: Eq. (7) itself, brute force over
all K-subsets, scipy's softmax and logsumexp, closed cases.  Then mistakes
planted in copies of the oracle must each fail one of these pins."""
import itertools
import types

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

import oracle.readout as RO


def _rows(seed, R, V, scale):
    return np.random.default_rng(seed).normal(0.0, scale, size=(R, V)).astype(np.float32)


# ----------------------------------------------------------------- the pins
def pin_eq7_total_variation(ro):
    # Eq. (7): renormalising the returned set moves the distribution by
    # exactly the omitted mass, TV(p, q) = 1 - Z
    for seed, V, k, scale in ((1, 50, 5, 1.0), (2, 300, 17, 3.0), (3, 64, 64, 0.5), (4, 1000, 256, 2.0)):
        x = _rows(seed, 3, V, scale)
        ids, probs, z, lse = ro.readout_topk(x, k)
        p_full = softmax(x.astype(np.float64), axis=1)
        for r in range(3):
            q = RO.renormalised(p_full[r], ids[r])
            assert abs(RO.total_variation(p_full[r], q) - (1.0 - z[r])) < 1e-12


def pin_topk_maximises_retained_mass(ro):
    # brute force: no other K-subset keeps more probability than the returned one
    x = _rows(5, 4, 9, 1.5)
    p = softmax(x.astype(np.float64), axis=1)
    for k in (1, 3, 5):
        ids, probs, z, _ = ro.readout_topk(x, k)
        for r in range(4):
            best = max(p[r, list(c)].sum() for c in itertools.combinations(range(9), k))
            assert abs(z[r] - best) < 1e-12
            assert len(set(ids[r].tolist())) == k


def pin_probs_are_the_full_distribution(ro):
    # probabilities of the full softmax (scipy), in descending order, and
    # their sum is Z
    x = _rows(6, 5, 777, 2.5)
    ids, probs, z, lse = ro.readout_topk(x, 40)
    p = softmax(x.astype(np.float64), axis=1)
    for r in range(5):
        assert np.allclose(probs[r], p[r, ids[r]], rtol=1e-12, atol=0)
        assert np.all(np.diff(probs[r]) <= 0)
        assert abs(probs[r].sum() - z[r]) < 1e-12
    assert np.allclose(lse, logsumexp(x.astype(np.float64), axis=1), rtol=1e-13, atol=0)


def pin_closed_cases(ro):
    x = _rows(7, 3, 33, 1.0)
    _, _, z, _ = ro.readout_topk(x, 33)          # K = V keeps everything
    assert np.allclose(z, 1.0, atol=1e-12)
    ids, _, _, _ = ro.readout_topk(x, 1)         # K = 1 is the argmax
    assert np.array_equal(ids[:, 0], np.argmax(x, axis=1))
    # equal logits: smaller token id first
    t = np.array([[1.0, 3.0, 3.0, 0.0, 3.0, -2.0]], np.float32)
    assert ro.readout_topk(t, 2)[0].tolist() == [[1, 2]]
    assert ro.readout_topk(t, 4)[0].tolist() == [[1, 2, 4, 0]]
    # a constant added to every logit changes nothing (softmax shift
    # invariance; the shift is exact in float64)
    a = ro.readout_topk(x, 7)
    b = ro.readout_topk(x.astype(np.float64) + 100.0, 7)
    assert np.array_equal(a[0], b[0]) and np.allclose(a[1], b[1], rtol=1e-12)
    # masked tokens (-inf) carry no probability and come last
    m = np.array([[0.5, -np.inf, 2.0, -np.inf]], np.float32)
    ids, probs, z, _ = ro.readout_topk(m, 3)
    assert ids.tolist() == [[2, 0, 1]] and probs[0, 2] == 0.0 and abs(z[0] - 1.0) < 1e-12
    # large logits stay finite
    big = np.array([[1e4, -1e4, 9990.0]], np.float32)
    ids, probs, z, lse = ro.readout_topk(big, 2)
    assert np.all(np.isfinite(probs)) and np.isfinite(lse[0]) and ids.tolist() == [[0, 2]]


PINS = [pin_eq7_total_variation, pin_topk_maximises_retained_mass,
        pin_probs_are_the_full_distribution, pin_closed_cases]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_readout_oracle_pins(pin):
    pin(RO)


# ------------------------------------------------------- planted mistakes
MUTANTS = {
    "ascending_order": ("np.lexsort((tok, -x[r]))", "np.lexsort((tok, x[r]))"),
    "ties_larger_id_first": ("np.lexsort((tok, -x[r]))", "np.lexsort((-tok, -x[r]))"),
    "renormalised_probs": ("probs[r] = np.exp(x[r, order] - lse[r])",
                           "probs[r] = np.exp(x[r, order] - lse[r]); probs[r] /= probs[r].sum()"),
    "one_too_few": ("[:k]\n", "[:k - 1]\n"),
    "max_not_subtracted": ("lse = m + np.log(np.exp(x - m[:, None]).sum(axis=1))",
                           "lse = np.log(np.exp(x - m[:, None]).sum(axis=1))"),
    "log2_normaliser": ("lse = m + np.log(np.exp(x - m[:, None]).sum(axis=1))",
                        "lse = m + np.log2(np.exp(x - m[:, None]).sum(axis=1))"),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_mistakes_fail_a_pin(name):
    src = open(RO.__file__).read()
    a, b = MUTANTS[name]
    assert src.count(a) >= 1, name
    mod = types.ModuleType("readout_mutant")
    exec(compile(src.replace(a, b), "readout_mutant", "exec"), mod.__dict__)
    failed = 0
    for pin in PINS:
        try:
            pin(mod)
        except (AssertionError, ValueError, IndexError):
            failed += 1
    assert failed > 0, f"mutant {name} passed every pin"
