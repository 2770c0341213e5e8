"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every function include/pie_fwd.h declares, and its planner's
metadata validation agrees with the oracle's on valid and invalid passes."""
import ctypes as C

import numpy as np
import pytest

import oracle as O
import workloads as W
from programmable_paged_kv_gb300 import abi, build, make_desc, make_meta


@pytest.fixture(scope="module")
def lib():
    build()
    return abi.load()


def test_library_exports_every_header_function(lib):
    names = abi.header_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
        assert n in abi.SIGNATURES, n


def test_build_can_be_called_again(lib):
    # the package's build() stays the function after its builder module loads
    import programmable_paged_kv_gb300 as pk
    assert callable(pk.build)
    pk.build()
    assert callable(pk.build)


def test_abi_version(lib):
    assert lib.pie_fwd_abi_version() == 105


def test_timing_events_need_both_or_neither(lib):
    assert lib.pie_fwd_set_timing_events(C.c_void_p(1), None) != 0
    assert lib.pie_fwd_set_timing_events(None, None) == 0


def _ws(desc, p, num_pool_pages):
    n = C.c_size_t(0)
    m = make_meta(p, num_pool_pages)
    rc = abi.load().pie_fwd_workspace_bytes(C.byref(make_desc(desc)), C.byref(m.c), C.byref(n))
    return rc, int(n.value)


@pytest.mark.parametrize("name", W.SMALL_NAMES)
def test_valid_scenarios_plan_on_host(lib, name):
    sc = W.small(name, 0)
    for p in sc.passes:
        rc, n = _ws(sc.desc, p, sc.num_pool_pages)
        assert rc == abi.PIE_OK, lib.pie_fwd_last_error()
        assert n > 0 and n % 256 == 0


def _base():
    desc = W.Desc(4, 2, 64, 16, W.BF16)
    z = np.zeros((2, 4, 64), np.uint16)
    zk = np.zeros((2, 2, 64), np.uint16)
    p = W.Pass(row_indptr=np.array([0, 2], np.int32), positions=np.array([20, 21], np.int32),
               slots=np.array([20, 21], np.int32), kv_len=np.array([22], np.int32),
               page_indptr=np.array([0, 2], np.int32), page_ids=np.array([3, 1], np.int32),
               fold_mode=np.array([W.FOLD_ALL], np.int32), fold_count=np.zeros(1, np.int32),
               q=z, k=zk, v=zk)
    return desc, p


def _set(**kw):
    def f(p):
        for k, v in kw.items():
            setattr(p, k, v)
    return f


CASES = [
    ("ok", lambda p: None),
    ("indptr_end", _set(row_indptr=np.array([0, 3], np.int32))),
    ("indptr_start", _set(row_indptr=np.array([1, 2], np.int32))),
    ("slot_past_pages", _set(slots=np.array([20, 32], np.int32))),
    ("negative_slot", _set(slots=np.array([-1, 21], np.int32), fold_mode=np.array([0], np.int32))),
    ("negative_position", _set(positions=np.array([-5, 21], np.int32))),
    ("kv_len_past_pages", _set(kv_len=np.array([33], np.int32))),
    ("negative_kv_len", _set(kv_len=np.array([-1], np.int32))),
    ("page_outside_pool", _set(page_ids=np.array([3, 4], np.int32))),
    ("fold_non_consecutive", _set(slots=np.array([21, 20], np.int32))),
    ("duplicate_target", _set(slots=np.array([21, 21], np.int32), fold_mode=np.array([0], np.int32))),
    ("unknown_fold", _set(fold_mode=np.array([9], np.int32))),
    ("fold_count_range", _set(fold_mode=np.array([2], np.int32), fold_count=np.array([3], np.int32))),
    ("fold_count_ok", _set(fold_mode=np.array([2], np.int32), fold_count=np.array([2], np.int32))),
    ("readout_range", _set(readout=np.array([0, 2], np.int32))),
    ("readout_ok", _set(readout=np.array([1, 0, 1], np.int32))),
    ("mask_too_short", _set(mask_word_indptr=np.array([0, 1, 1], np.int64))),
    ("mask_ok", _set(mask_word_indptr=np.array([0, 1, 2], np.int64))),
    ("mask_decreasing", _set(mask_word_indptr=np.array([0, 2, 1], np.int64))),
]


@pytest.mark.parametrize("name,mutate", CASES, ids=[c[0] for c in CASES])
def test_validation_agrees_with_oracle(lib, name, mutate):
    desc, p = _base()
    mutate(p)
    rc_lib, _ = _ws(desc, p, 4)
    rc_orc = O.validate(desc, p, num_pool_pages=4)
    assert rc_lib == rc_orc, (name, rc_lib, rc_orc, lib.pie_fwd_last_error())


def test_unsupported_shapes_are_refused(lib):
    _, p = _base()
    for desc in (W.Desc(4, 2, 96, 16, W.BF16), W.Desc(4, 2, 64, 12, W.BF16),
                 W.Desc(32, 2, 64, 16, W.BF16)):
        rc, _ = _ws(desc, p, 4)
        assert rc == abi.PIE_EUNSUPPORTED
    rc, _ = _ws(W.Desc(4, 3, 64, 16, W.BF16), p, 4)
    assert rc == abi.PIE_EINVAL


def test_empty_pass_plans(lib):
    desc = W.Desc(4, 2, 64, 16, W.BF16)
    e = np.zeros(0, np.int32)
    z = np.zeros((0, 4, 64), np.uint16)
    p = W.Pass(row_indptr=np.zeros(1, np.int32), positions=e, slots=e, kv_len=e,
               page_indptr=np.zeros(1, np.int32), page_ids=e, fold_mode=e, fold_count=e,
               q=z, k=z, v=z)
    rc, n = _ws(desc, p, 0)
    assert rc == abi.PIE_OK and n >= 0


def test_readout_refuses_bad_calls_before_any_launch(lib):
    n = C.c_size_t(0)
    ws = lib.pie_fwd_readout_topk_workspace_bytes
    assert ws(abi.PIE_F32, 64, 128256, 256, C.byref(n)) == abi.PIE_OK and n.value > 0
    assert ws(abi.PIE_F32, 4, 1000, 0, C.byref(n)) == abi.PIE_EINVAL        # k < 1
    assert ws(abi.PIE_F32, 4, 100, 101, C.byref(n)) == abi.PIE_EINVAL       # k > vocab
    assert ws(7, 4, 1000, 8, C.byref(n)) == abi.PIE_EINVAL                  # dtype
    assert ws(abi.PIE_F32, 4, 1000, 257, C.byref(n)) == abi.PIE_EUNSUPPORTED
    assert ws(abi.PIE_BF16, 4, 262145, 8, C.byref(n)) == abi.PIE_EUNSUPPORTED
    assert ws(abi.PIE_BF16, 4, 262144, 8, C.byref(n)) == abi.PIE_OK
    # rows that do not start on 16-byte boundaries (fp32, ld 1001) and a NULL
    # output are refused before anything is launched (the pointers are never
    # dereferenced)
    p = C.c_void_p(4096)
    assert lib.pie_fwd_readout_topk(p, abi.PIE_F32, 2, 1001, 1001, 8, p, p, None, None, p, 1 << 20,
                                    None) == abi.PIE_EINVAL
    assert lib.pie_fwd_readout_topk(p, abi.PIE_F32, 2, 1000, 1000, 8, None, p, None, None, p, 1 << 20,
                                    None) == abi.PIE_EINVAL
    assert lib.pie_fwd_readout_topk(p, abi.PIE_F32, 2, 1000, 1000, 8, p, p, None, None, p, 16,
                                    None) == abi.PIE_ENOSPACE


def test_adapter_plan_refuses_bad_lanes_before_any_cuda_call(lib):
    i32 = lambda a: np.ascontiguousarray(a, dtype=np.int32)
    n = C.c_size_t(0)
    ws = lib.pie_fwd_adapter_workspace_bytes
    ri = i32([0, 1, 130, 130, 131])
    assert ws(4, ri.ctypes.data, 16, C.byref(n)) == abi.PIE_OK
    # tiles: 1 + 2 + 0 + 1 rows-of-128 blocks, 16 bytes each, and a counter
    # each (256-aligned); groups of the grouped path (at most one per tile,
    # 16 bytes each) and their rows (131 int32); then 8 ranges x 131 rows x 16
    # fp32 partial sums and 131 x 16 final sums
    up = lambda v: (v + 255) // 256 * 256
    assert n.value == 256 + 256 + 256 + up(131 * 4) + up(8 * 131 * 16 * 4) + up(131 * 16 * 4)
    assert ws(4, ri.ctypes.data, 12, C.byref(n)) == abi.PIE_EUNSUPPORTED   # rank not built
    assert ws(2, i32([0, 3, 2]).ctypes.data, 16, C.byref(n)) == abi.PIE_EINVAL   # not monotone
    assert ws(1, i32([1, 3]).ctypes.data, 16, C.byref(n)) == abi.PIE_EINVAL      # indptr[0] != 0
    h = C.c_void_p()
    plan = lib.pie_fwd_adapter_plan
    ad = i32([0, 1, -1, 2])
    buf = C.c_void_p(1 << 20)   # never dereferenced: every call below fails validation first
    assert plan(4, ri.ctypes.data, i32([0, 3, -1, 2]).ctypes.data, 3, 16, buf, 1 << 30, None,
                C.byref(h)) == abi.PIE_ERANGE                                   # adapter 3 of 3
    assert plan(4, ri.ctypes.data, i32([0, -2, -1, 2]).ctypes.data, 3, 16, buf, 1 << 30, None,
                C.byref(h)) == abi.PIE_ERANGE                                   # adapter -2
    assert plan(4, ri.ctypes.data, ad.ctypes.data, 3, 16, buf, 16, None,
                C.byref(h)) == abi.PIE_ENOSPACE
    assert plan(4, ri.ctypes.data, ad.ctypes.data, 3, 16, C.c_void_p((1 << 20) + 16), 1 << 30,
                None, C.byref(h)) == abi.PIE_EINVAL                             # alignment
    assert plan(4, ri.ctypes.data, None, 3, 16, buf, 1 << 30, None, C.byref(h)) == abi.PIE_EINVAL
    assert h.value is None
    apply = lib.pie_fwd_adapter_apply
    assert apply(None, abi.PIE_BF16, 64, 256, 16, buf, buf, buf, buf, buf, None, None,
                 None) == abi.PIE_EINVAL
