"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.

* every small scenario (several KV tiles, ragged lanes and tails) compared
  element by element: pools, q_rot, outputs and lse of every row, readout
  rows, frozen lengths and status words;
* the full-size configurations, in the launch configuration the benchmark
  times, compared on sampled rows (the oracle computes those rows only) plus
  every bookkeeping result, and the full guidance-pair configuration on every
  row (all 4,096 prefill rows of the tensor-core path);
* edge cases: empty passes, lanes without rows, empty visible sets, frozen
  writes, clamped channel counts, fold gaps, other head sizes, page sizes
  and fp32.
"""
import os

import numpy as np
import pytest

import oracle as O
import workloads as W
from tests.parity import compare_scenario

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

THREADS = max(1, (os.cpu_count() or 2) - 1)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from programmable_paged_kv_gb300 import abi, build
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build()
    abi.load()


def _run_both(sc, rows_per_pass=None):
    from programmable_paged_kv_gb300 import runner
    gpu = runner.run_scenario(sc)
    orc = O.run_scenario(sc, num_threads=THREADS, rows_per_pass=rows_per_pass)
    return gpu, orc


@pytest.mark.parametrize("seed", [0, 1])
@pytest.mark.parametrize("name", W.SMALL_NAMES)
def test_small_scenario_matches_oracle(name, seed):
    sc = W.small(name, seed)
    gpu, orc = _run_both(sc)
    compare_scenario(sc, gpu, orc)


def _sample_rows(p, per_lane, rng):
    rows = []
    for l in range(p.num_lanes):
        r0, r1 = int(p.row_indptr[l]), int(p.row_indptr[l + 1])
        if r1 > r0:
            k = min(per_lane, r1 - r0)
            rows.extend(sorted(set([r1 - 1] + list(rng.choice(np.arange(r0, r1), k, replace=False)))))
    return np.array(sorted(set(rows)), np.int32)


FULL_SAMPLING = {  # rows per lane the oracle recomputes, per pass kind
    "tiny": None,
    "decode_batch": None,
    "guidance_pairs": 1,
    "spec_verify": 1,
    "masked_window": 2,
    "masked_tova": 1,
    "masked_decode_window": None,
    "masked_decode_tova": None,
}


@pytest.mark.parametrize("name", list(W.FULL.keys()))
def test_full_size_configuration_sampled(name):
    sc = W.FULL[name](0)
    per_lane = FULL_SAMPLING[name]
    rows = None
    if per_lane is not None:
        rng = np.random.default_rng(123)
        rows = [_sample_rows(p, per_lane, rng) if p.num_rows > p.num_lanes else None
                for p in sc.passes]
        # decode passes of the guidance scenario: every row (one per lane)
    gpu, orc = _run_both(sc, rows)
    compare_scenario(sc, gpu, orc, rows)


def test_full_size_guidance_prefill_every_row():
    """The full guidance-pair configuration (64 lanes x 64 prefill rows on a
    shared 1,024-slot prefix, then 16 decode passes) with every row of every
    pass recomputed by the oracle: all 4,096 prefill rows of the tensor-core
    path, not a sample."""
    sc = W.FULL["guidance_pairs"](0)
    gpu, orc = _run_both(sc)
    compare_scenario(sc, gpu, orc)


VARIANTS = {
    "d64_p8_bf16": W.Desc(8, 2, 64, 8, W.BF16),
    "d64_p32_bf16": W.Desc(8, 2, 64, 32, W.BF16),
    "d128_p32_f32": W.Desc(8, 4, 128, 32, W.F32),
    "d64_p16_f32": W.Desc(4, 4, 64, 16, W.F32),
    "g8_d128_p16_bf16": W.Desc(16, 2, 128, 16, W.BF16),
    "g1_d128_p16_bf16": W.Desc(4, 4, 128, 16, W.BF16),
}


@pytest.mark.parametrize("var", list(VARIANTS))
def test_shape_variants(var):
    desc = VARIANTS[var]
    for sc in (W.decode_batch(3, lanes=5, c_lo=1, c_hi=300, num_pool_pages=400, desc=desc),
               W.guidance_pairs(3, pairs=2, prefix=64, prefill=9, decodes=2, num_pool_pages=64,
                                desc=desc),
               W.spec_verify(3, lanes=3, draft=5, c_lo=30, c_hi=200, num_pool_pages=128, desc=desc)):
        gpu, orc = _run_both(sc)
        compare_scenario(sc, gpu, orc)


# Masked passes on the tensor-core path: window masks (the pre-pass lists
# whole pages) and TOVA masks (it lists single slots), one and two query
# tiles per item, every page size, the last page cut by kv_len.
MASKED_VARIANTS = {
    "window_one_tile_p8": (W.Desc(32, 8, 128, 8, W.BF16),
                           dict(kind="window", lanes=2, kv=700, rows=24, window=200)),
    "window_two_tiles_p32": (W.Desc(32, 8, 128, 32, W.BF16),
                             dict(kind="window", lanes=2, kv=1000, rows=40, window=250)),
    "tova_one_tile_p16": (W.Desc(32, 8, 128, 16, W.BF16),
                          dict(kind="tova", lanes=2, kv=900, rows=24)),
    "window_g1_two_tiles_p16": (W.Desc(8, 8, 128, 16, W.BF16),
                                dict(kind="window", lanes=2, kv=777, rows=150, window=200)),
    # decode rows (one or two per lane, G = 4 and 8): fewer than 16 query
    # vectors per kv head, served by the tensor-core kernel's compacted lists
    "window_decode_p16": (W.Desc(32, 8, 128, 16, W.BF16),
                          dict(kind="window", lanes=3, kv=2000, rows=1, window=500)),
    "tova_decode_p8": (W.Desc(32, 8, 128, 8, W.BF16),
                       dict(kind="tova", lanes=3, kv=1500, rows=1)),
    "window_two_rows_g8_p32": (W.Desc(16, 2, 128, 32, W.BF16),
                               dict(kind="window", lanes=2, kv=1700, rows=2, window=333)),
}


@pytest.mark.parametrize("var", list(MASKED_VARIANTS))
def test_masked_list_modes(var):
    desc, kw = MASKED_VARIANTS[var]
    sc = W.masked_long(5, desc=desc, **kw)
    gpu, orc = _run_both(sc)
    compare_scenario(sc, gpu, orc)


def test_set_mask_lists_serve_every_layer():
    """pie_fwd_set_mask builds a pass's compacted lists once; attend on two
    layers (two pairs of pools, the same mask) reuses them and returns what
    a plan that builds its own lists at every attend returns, bit for bit."""
    import torch
    from programmable_paged_kv_gb300 import ForwardPlan, make_desc, make_meta, runner
    for sc in (W.small("masked_window", 2), W.small("masked_decode_tova", 2)):
        d, p = sc.desc, sc.passes[0]
        desc = make_desc(d)
        layers = [runner.DevicePools(sc), runner.DevicePools(sc)]
        # the second layer's cached K/V differ from the first's
        g = torch.Generator(device="cuda").manual_seed(5)
        for t in (layers[1].k, layers[1].v):
            t.index_copy_(0, layers[1].used, torch.randn(
                (layers[1].used.numel(),) + tuple(t.shape[1:]), generator=g,
                device="cuda").to(t.dtype))
        N, Hq, D = p.num_rows, d.num_q_heads, d.head_dim
        mw = torch.from_numpy(p.mask_words.view(np.int32)).cuda()
        q_rot = torch.empty((N, Hq, D), dtype=torch.bfloat16, device="cuda")
        outs = {}
        for mode in ("set_mask", "per_call"):
            plan = ForwardPlan(desc, make_meta(p, sc.num_pool_pages))
            frozen = torch.from_numpy(sc.frozen_len0.astype(np.int32)).cuda()
            q, k, v = (runner.to_device(x, d.dtype) for x in (p.q, p.k, p.v))
            if mode == "set_mask":
                plan.set_mask(mw)
            for li, pools in enumerate(layers):
                kk, vv = pools.k.clone(), pools.v.clone()
                plan.append_kv(q, k, v, q_rot, kk, vv, frozen)
                o = torch.empty((N, Hq, D), dtype=torch.bfloat16, device="cuda")
                lse = torch.empty((N, Hq), dtype=torch.float32, device="cuda")
                ro = torch.empty((plan.num_readout, Hq, D), dtype=torch.bfloat16, device="cuda")
                plan.attend(q_rot, kk, vv, mw, ro, None, o, lse)
                outs[(mode, li)] = (o.view(torch.int16).cpu(), lse.cpu())
            torch.cuda.synchronize()
            plan.close()
        for li in range(2):
            a, b = outs[("set_mask", li)], outs[("per_call", li)]
            assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
        assert not torch.equal(outs[("set_mask", 0)][0], outs[("set_mask", 1)][0])


# ---------------------------------------------------------------- edge cases
def _one_pass_scenario(desc, p, frozen0, pool_pages_n, fill_slots):
    """Scenario around one hand-made pass; fill_slots[l] cached slots random."""
    rng = np.random.default_rng(7)
    lane_pages = [p.page_ids[p.page_indptr[l]:p.page_indptr[l + 1]] for l in range(p.num_lanes)]
    pool_pages = np.unique(p.page_ids).astype(np.int32)
    k0, v0 = W._fill_pool_init(desc, pool_pages, lane_pages, fill_slots, rng)
    return W.Scenario("edge", desc, pool_pages_n, pool_pages, k0, v0,
                      np.asarray(frozen0, np.int32), [p])


def _mk_pass(desc, lanes, rng, fold=W.FOLD_ALL, masks=None, readout=None, channel=None):
    """lanes: list of (kv_len, [(pos, slot), ...], pages)."""
    rows = [([r[0] for r in rs], [r[1] for r in rs]) for _, rs, _ in lanes]
    return W._lane_pass(desc, rows, [pg for _, _, pg in lanes], [kv for kv, _, _ in lanes],
                        [fold] * len(lanes), rng, mask_rows=masks, readout=readout,
                        channel=channel)


def test_empty_pass_and_lanes_without_rows():
    desc = W.Desc(8, 2, 128, 16, W.BF16)
    rng = np.random.default_rng(1)
    lanes = [(40, [(39, 39)], [0, 1, 2]), (0, [], [3]), (20, [], [4, 5]), (17, [(16, 16)], [6, 7])]
    p = _mk_pass(desc, lanes, rng)
    sc = _one_pass_scenario(desc, p, [39, 0, 20, 16], 8, [39, 0, 20, 16])
    gpu, orc = _run_both(sc)
    compare_scenario(sc, gpu, orc)
    assert gpu[3][0]["out_readout"].shape[0] == 2
    # a pass with no lanes at all
    e = np.zeros(0, np.int32)
    z = np.zeros((0, 8, 128), np.uint16)
    z2 = np.zeros((0, 2, 128), np.uint16)
    p0 = W.Pass(row_indptr=np.zeros(1, np.int32), positions=e, slots=e, kv_len=e,
                page_indptr=np.zeros(1, np.int32), page_ids=e, fold_mode=e, fold_count=e,
                q=z, k=z2, v=z2)
    sc0 = W.Scenario("empty", desc, 1, np.zeros(0, np.int32), np.zeros((0, 2, 16, 128), np.uint16),
                     np.zeros((0, 2, 16, 128), np.uint16), np.zeros(0, np.int32), [p0])
    from programmable_paged_kv_gb300 import runner
    _, _, fr, res, ok = runner.run_scenario(sc0)
    assert res[0]["out_readout"].shape[0] == 0 and ok


def test_empty_visible_sets_give_zero_and_minus_inf():
    desc = W.Desc(8, 2, 128, 16, W.BF16)
    rng = np.random.default_rng(2)
    kv = 70
    lanes = [(kv, [(68, 68), (69, 69)], [0, 1, 2, 3, 4]), (0, [(0, 0)], [5])]
    masks = [np.zeros(kv, bool), np.r_[np.zeros(kv - 1, bool), True], np.zeros(0, bool)]
    p = _mk_pass(desc, lanes, rng, fold=W.FOLD_NONE, masks=masks)
    sc = _one_pass_scenario(desc, p, [68, 0], 6, [68, 0])
    gpu, orc = _run_both(sc)
    compare_scenario(sc, gpu, orc)
    lse = gpu[3][0]["lse_all"]
    assert np.isneginf(lse[0]).all() and np.isneginf(lse[2]).all() and np.isfinite(lse[1]).all()


def test_frozen_write_fold_gap_and_channel_clamp_status():
    desc = W.Desc(8, 2, 64, 16, W.BF16)
    rng = np.random.default_rng(3)
    # lane 0 writes into its frozen prefix (slot 5 < 10); lane 1 folds from a
    # channel value out of range; lane 2's first slot is past its frozen length
    lanes = [(12, [(10, 10), (11, 11)], [0]), (12, [(10, 10), (11, 11)], [1]),
             (14, [(12, 12), (13, 13)], [2])]
    p = _mk_pass(desc, lanes, rng, fold=W.FOLD_CHANNEL, channel=[1, 9, -3])
    p.slots = np.array([5, 6, 10, 11, 12, 13], np.int32)
    p.positions = p.slots.copy()
    # lane 2 holds finite K/V in slot 11 (read by its rows) although only
    # slots below 11 are frozen
    sc = _one_pass_scenario(desc, p, [10, 10, 11], 3, [10, 10, 12])
    gpu, orc = _run_both(sc)
    compare_scenario(sc, gpu, orc)
    st = gpu[3][0]["status"]
    assert st & O.ST_FROZEN_WRITE and st & O.ST_FOLD_CLAMP and st & O.ST_FOLD_GAP


def test_readout_list_with_repeats():
    sc = W.small("spec_verify", 4)
    p = sc.passes[0]
    p.readout = np.array([3, 0, 3, p.num_rows - 1, 7], np.int32)
    gpu, orc = _run_both(sc)
    compare_scenario(sc, gpu, orc)


def test_invalid_calls_are_refused_without_launch():
    from programmable_paged_kv_gb300 import ForwardPlan, PieError, abi, make_desc, make_meta
    sc = W.small("decode_batch", 0)
    p = sc.passes[0]
    plan = ForwardPlan(make_desc(sc.desc), make_meta(p, sc.num_pool_pages))
    q = torch.zeros(1, device="cuda")
    with pytest.raises(PieError) as e:
        plan.attend(q, q, q, mask_words=q.int())  # the plan has no mask
    assert e.value.code == abi.PIE_EINVAL
    with pytest.raises(PieError) as e:
        plan.append_kv(q, q, q, None, q, q, q)
    assert e.value.code == abi.PIE_EINVAL
    torch.cuda.synchronize()
    plan.close()
    sc = W.small("spec_verify", 0)
    plan = ForwardPlan(make_desc(sc.desc), make_meta(sc.passes[0], sc.num_pool_pages))
    with pytest.raises(PieError) as e:
        plan.fold(torch.zeros(sc.passes[0].num_lanes, dtype=torch.int32, device="cuda"), None)
    assert e.value.code == abi.PIE_EINVAL
    plan.close()
