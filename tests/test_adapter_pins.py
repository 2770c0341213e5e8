"""Pins of the adapter oracle (Pie "The forward pass", Adapters: LoRA
y + b (a x), IA3 y scaled, a different adapter per lane) against facts fixed
outside it: explicit loops on tiny shapes, closed cases, linearity; then
mistakes planted in copies of the oracle must each fail a pin."""
import types

import numpy as np
import pytest

import oracle.adapters as AD


def _case(seed, L=3, rows=(2, 0, 3), d_in=5, d_out=4, r=2, n_ad=2, ia3=True):
    g = np.random.default_rng(seed)
    row_indptr = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    N = int(row_indptr[-1])
    x = g.normal(size=(N, d_in))
    y = g.normal(size=(N, d_out))
    A = g.normal(size=(n_ad, r, d_in))
    B = g.normal(size=(n_ad, d_out, r))
    scale = g.uniform(0.5, 2.0, size=n_ad)
    s = g.uniform(0.5, 1.5, size=(n_ad, d_out)) if ia3 else None
    lane_ad = np.array([1, 0, -1][:L], np.int32)
    return x, y, row_indptr, lane_ad, A, B, scale, s


def pin_explicit_loops(ad):
    # every output element written out as sums over the rank and the input
    x, y, ri, la, A, B, sc, s = _case(1)
    got = ad.apply_adapters(x, y, ri, la, A, B, sc, s)
    for l in range(len(la)):
        for row in range(ri[l], ri[l + 1]):
            for o in range(y.shape[1]):
                want = y[row, o]
                a = la[l]
                if a >= 0:
                    acc = 0.0
                    for k in range(A.shape[1]):
                        acc += B[a, o, k] * sum(A[a, k, i] * x[row, i] for i in range(x.shape[1]))
                    want = (want + sc[a] * acc) * s[a, o]
                assert abs(got[row, o] - want) < 1e-12


def pin_closed_cases(ad):
    x, y, ri, la, A, B, sc, s = _case(2, ia3=False)
    # no adapter on any lane, or a zero B, leaves y as it is
    assert np.array_equal(ad.apply_adapters(x, y, ri, np.full(3, -1, np.int32), A, B, sc, None), y)
    assert np.array_equal(ad.apply_adapters(x, y, ri, la, A, np.zeros_like(B), sc, None), y)
    # IA3 alone (LoRA scale 0) scales y elementwise
    s = np.random.default_rng(3).uniform(0.5, 1.5, size=(2, y.shape[1]))
    got = ad.apply_adapters(x, y, ri, la, A, B, np.zeros(2), s)
    assert np.allclose(got[0:2], y[0:2] * s[1], rtol=1e-14)
    assert np.array_equal(got[2:], y[2:])
    # rank one with unit vectors: y'[o] = y[o] + scale * x[i]
    A1 = np.zeros((2, 1, x.shape[1])); A1[:, 0, 3] = 1.0
    B1 = np.zeros((2, y.shape[1], 1)); B1[:, 2, 0] = 1.0
    got = ad.apply_adapters(x, y, ri, la, A1, B1, np.array([0.5, 2.0]), None)
    want = y.copy()
    want[0:2, 2] += 2.0 * x[0:2, 3]   # lane 0 uses adapter 1
    assert np.allclose(got, want, rtol=0, atol=1e-14)
    # linear in the scale: the change at 2 * scale is twice the change at scale
    d1 = ad.apply_adapters(x, y, ri, la, A, B, sc, None) - y
    d2 = ad.apply_adapters(x, y, ri, la, A, B, 2 * sc, None) - y
    assert np.allclose(d2, 2 * d1, rtol=1e-12, atol=1e-12)


PINS = [pin_explicit_loops, pin_closed_cases]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_adapter_oracle_pins(pin):
    pin(AD)


MUTANTS = {
    "A_not_transposed": ("x[r0:r1] @ np.asarray(A[a], np.float64).T", "x[r0:r1] @ np.asarray(A[a], np.float64).T[::-1]"),
    "scale_dropped": ("float(scale[a]) * (t @", "1.0 * (t @"),
    "ia3_before_lora": ("yl = out[r0:r1] + float(scale[a]) * (t @ np.asarray(B[a], np.float64).T)\n        if ia3 is not None:\n            yl = yl * np.asarray(ia3[a], np.float64)[None, :]",
                        "yl = out[r0:r1]\n        if ia3 is not None:\n            yl = yl * np.asarray(ia3[a], np.float64)[None, :]\n        yl = yl + float(scale[a]) * (t @ np.asarray(B[a], np.float64).T)"),
    "wrong_lane_rows": ("r0, r1 = int(row_indptr[l]), int(row_indptr[l + 1])", "r0, r1 = int(row_indptr[l]), int(row_indptr[l + 1]) + 1"),
    "none_lane_applied": ("if a < 0 or r1 == r0:", "if r1 == r0:"),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_mistakes_fail_a_pin(name):
    src = open(AD.__file__).read()
    a, b = MUTANTS[name]
    assert src.count(a) >= 1, name
    mod = types.ModuleType("adapters_mutant")
    exec(compile(src.replace(a, b), "adapters_mutant", "exec"), mod.__dict__)
    failed = 0
    for pin in PINS:
        try:
            pin(mod)
        except (AssertionError, ValueError, IndexError):
            failed += 1
    assert failed > 0, f"mutant {name} passed every pin"
