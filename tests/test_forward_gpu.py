"""pie_fwd_forward (plan, append_kv, set_mask, attend and fold of one pass in
one call) against the same pass run call by call: the same kernels on the
same inputs in the same order, so every output, the pools and the frozen
lengths must agree bit for bit, on every small scenario (masked passes,
channel folds, decode, prefill, verify)."""
import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from programmable_paged_kv_gb300 import build
    build()


@pytest.mark.parametrize("name", W.SMALL_NAMES)
def test_one_call_equals_the_calls(name):
    from programmable_paged_kv_gb300 import runner
    sc = W.small(name, 0)
    k_a, v_a, fr_a, res_a, ok_a = runner.run_scenario(sc)
    k_b, v_b, fr_b, res_b, ok_b = runner.run_scenario(sc, one_call=True)
    assert ok_a and ok_b
    assert np.array_equal(k_a, k_b) and np.array_equal(v_a, v_b) and np.array_equal(fr_a, fr_b)
    for i, (a, b) in enumerate(zip(res_a, res_b)):
        for key in a:
            assert np.array_equal(np.asarray(a[key]), np.asarray(b[key])), (name, i, key)
