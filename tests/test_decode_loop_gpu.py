"""Decode loop that runs ahead of the host (pie_fwd_decode_loop; Pie "The
forward pass", Pipelines and frames: run_ahead) against the oracle run pass
by pass on the same inputs: every step's output and lse, the K/V pools, the
frozen lengths and the status word; pages outside the working sets stay
untouched; lanes with no slot left write nothing and return o = 0,
lse = -inf."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests.parity import (assert_bits_equal, assert_lse_close, assert_out_close,
                          assert_rope_close)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from programmable_paged_kv_gb300 import build
    build()


def _run_loop(sc, steps, frozen0=None, channel=None, page_ids=None):
    import torch
    from programmable_paged_kv_gb300 import decode_loop, make_desc, runner
    d = sc.desc
    desc = make_desc(d)
    pools = runner.DevicePools(sc)
    p0 = sc.passes[0]
    L, Hq, D = p0.num_lanes, d.num_q_heads, d.head_dim
    f0 = sc.frozen_len0 if frozen0 is None else frozen0
    frozen = torch.from_numpy(np.asarray(f0, np.int32)).cuda()
    page_indptr = torch.from_numpy(p0.page_indptr.astype(np.int32)).cuda()
    page_ids = torch.from_numpy(
        (p0.page_ids if page_ids is None else page_ids).astype(np.int32)).cuda()
    maxp = int(np.diff(p0.page_indptr).max())
    q = torch.stack([runner.to_device(sc.passes[t].q, d.dtype) for t in range(steps)])
    k = torch.stack([runner.to_device(sc.passes[t].k, d.dtype) for t in range(steps)])
    v = torch.stack([runner.to_device(sc.passes[t].v, d.dtype) for t in range(steps)])
    q_rot = torch.empty_like(q[0])
    out = torch.empty_like(q)
    lse = torch.empty((steps, L, Hq), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ch = None if channel is None else torch.from_numpy(np.asarray(channel, np.int32)).cuda()
    decode_loop(desc, page_indptr, page_ids, maxp, frozen, q, k, v, q_rot, pools.k, pools.v, out,
                lse, status, channel=ch)
    torch.cuda.synchronize()
    k_used = runner.to_host(pools.k.index_select(0, pools.used), d.dtype)
    v_used = runner.to_host(pools.v.index_select(0, pools.used), d.dtype)
    outs = [runner.to_host(out[t], d.dtype) for t in range(steps)]
    return (k_used, v_used, frozen.cpu().numpy(), outs, lse.cpu().numpy(), int(status.item()),
            runner._untouched_is_canary(pools, d.dtype))


VARIANTS = {
    "bf16_g4_p16": W.Desc(32, 8, 128, 16, W.BF16),
    "bf16_g8_p8_d64": W.Desc(16, 2, 64, 8, W.BF16),
    "f32_g2_p32": W.Desc(8, 4, 128, 32, W.F32),
}


@pytest.mark.parametrize("var", list(VARIANTS))
def test_decode_loop_matches_the_pass_by_pass_oracle(var):
    steps = 7
    sc = W.decode_loop(5, lanes=6, steps=steps, c_lo=1, c_hi=1500, num_pool_pages=900,
                       desc=VARIANTS[var])
    gk, gv, gfrozen, gouts, glse, gstatus, untouched = _run_loop(sc, steps)
    ok_, ov, ofrozen, ores = O.run_scenario(sc, num_threads=4)
    dt = sc.desc.dtype
    assert untouched, "a page outside the working sets was written"
    assert gstatus == 0
    assert np.array_equal(gfrozen, ofrozen)
    assert_rope_close(gk, ok_, dt, "K pool")
    assert_bits_equal(gv, ov, "V pool")
    for t in range(steps):
        assert_out_close(gouts[t], ores[t]["out"], dt, f"step {t} out")
        assert_lse_close(glse[t], ores[t]["lse"], dt, f"step {t} lse")


def test_lanes_without_a_free_slot_write_nothing():
    import torch  # noqa: F401
    sc = W.decode_loop(6, lanes=3, steps=2, c_lo=5, c_hi=60, num_pool_pages=64,
                       desc=W.Desc(8, 2, 64, 16, W.BF16))
    p0 = sc.passes[0]
    cap = np.diff(p0.page_indptr) * sc.desc.page_size
    gk, gv, gfrozen, gouts, glse, gstatus, untouched = _run_loop(sc, 2, frozen0=cap)
    assert gstatus & 64  # PIE_STATUS_LOOP_FULL
    assert np.array_equal(gfrozen, cap)          # nothing advanced
    assert untouched
    assert np.array_equal(gk, sc.k_init) and np.array_equal(gv, sc.v_init)  # nothing written
    for t in range(2):
        assert not np.any(gouts[t].astype(np.float64))
        assert np.all(np.isneginf(glse[t]))


def test_channel_fold_matches_the_pass_by_pass_oracle():
    """Step t folds clamp(channel[t][l], 0, 1): a lane given 0 keeps its frozen
    length, so its next step rewrites the same slot at the same position (the
    rejected token's K/V is overwritten, never read); counts outside [0, 1]
    (-1, 2, 7) are clamped and set PIE_STATUS_FOLD_CLAMP.  The oracle runs the
    same steps one pass at a time with the geometry each count implies."""
    steps, lanes = 8, 6
    sc = W.decode_loop(7, lanes=lanes, steps=steps, c_lo=1, c_hi=900, num_pool_pages=700,
                       desc=W.Desc(32, 8, 128, 16, W.BF16))
    rng = np.random.default_rng(11)
    channel = rng.choice([0, 1, 1, 1, -1, 2, 7], size=(steps, lanes)).astype(np.int32)
    gk, gv, gfrozen, gouts, glse, gstatus, untouched = _run_loop(sc, steps, channel=channel)
    # the oracle: step t at position = slot = F_t, kv_len F_t + 1, fold from
    # the channel (the oracle clamps and flags)
    k_pool, v_pool = sc.k_init.copy(), sc.v_init.copy()
    frozen = sc.frozen_len0.copy().astype(np.int32)
    ostatus = 0
    cp = sc.compact_page_ids(sc.passes[0].page_ids)
    for t in range(steps):
        p = sc.passes[t]
        F = frozen.copy()
        pt = W.Pass(p.row_indptr, F.copy(), F.copy(), (F + 1).astype(np.int32), p.page_indptr,
                    p.page_ids, np.full(lanes, W.FOLD_CHANNEL, np.int32), p.fold_count, p.q, p.k,
                    p.v, channel=channel[t])
        r = O.run_pass(sc.desc, pt, k_pool, v_pool, frozen, page_ids=cp, num_threads=4)
        assert r["err"] == O.OK
        ostatus |= r["status"]
        assert_out_close(gouts[t], r["out"], sc.desc.dtype, f"step {t} out")
        assert_lse_close(glse[t], r["lse"], sc.desc.dtype, f"step {t} lse")
    assert untouched
    assert np.array_equal(gfrozen, frozen)
    assert gstatus == ostatus and (gstatus & 2)  # PIE_STATUS_FOLD_CLAMP
    assert_rope_close(gk, k_pool, sc.desc.dtype, "K pool")
    assert_bits_equal(gv, v_pool, "V pool")


def test_out_of_pool_page_ids_are_skipped():
    """The loop's page table is device data: a page id outside the pool is
    neither written (RoPE/scatter) nor read (attention), PIE_STATUS_BOUNDS is
    set, nothing outside the working sets is touched, and the other lanes get
    the oracle's result."""
    steps, bad = 3, 1
    sc = W.decode_loop(8, lanes=4, steps=steps, c_lo=40, c_hi=300, num_pool_pages=256,
                       desc=W.Desc(8, 2, 128, 16, W.BF16))
    p0 = sc.passes[0]
    ids = p0.page_ids.copy()
    f = int(sc.frozen_len0[bad])
    ids[p0.page_indptr[bad] + f // sc.desc.page_size] = 1 << 28   # the page of its next slot
    ids[p0.page_indptr[bad]] = -5                                   # and its first page
    gk, gv, gfrozen, gouts, glse, gstatus, untouched = _run_loop(sc, steps, page_ids=ids)
    ok_, ov, ofrozen, ores = O.run_scenario(sc, num_threads=4)
    assert gstatus & 4  # PIE_STATUS_BOUNDS
    assert untouched
    good = [l for l in range(p0.num_lanes) if l != bad]
    assert np.array_equal(gfrozen, ofrozen)
    for t in range(steps):
        assert_out_close(gouts[t][good], ores[t]["out"][good], sc.desc.dtype, f"step {t} out")
        assert_lse_close(glse[t][good], ores[t]["lse"][good], sc.desc.dtype, f"step {t} lse")
