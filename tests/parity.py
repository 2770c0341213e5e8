"""Comparison helpers for GPU-vs-oracle parity tests.

Tolerances
  * integer / index / byte results (frozen lengths, status words, V payload
    written through the page table, untouched pages): bit-exact;
  * K pool and q_rot (RoPE results rounded to the dtype): within 1 ulp of
    bf16, or 2e-6 abs + 2e-6 rel for fp32 (the GPU evaluates the rotation in
    fp32, the oracle in double; both round once to the dtype);
  * attention output: bf16 max-abs 2e-2 and mean-abs 2e-3 (BF16 in, FP32
    accumulate, as the hot path's stated target); fp32 max-abs 1e-4 and
    mean-abs 1e-5;
  * lse (natural log): 2e-2 abs for bf16, 1e-4 for fp32; -inf exactly where
    the oracle has an empty visible set.
"""
import numpy as np

import workloads as W

OUT_TOL = {W.BF16: (2e-2, 2e-3), W.F32: (1e-4, 1e-5)}
LSE_TOL = {W.BF16: 2e-2, W.F32: 1e-4}


def bf16_ord(b: np.ndarray) -> np.ndarray:
    b = b.astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def _ulp(x: np.ndarray, mant_bits: int) -> np.ndarray:
    """Spacing of the dtype's numbers at |x| (normal range)."""
    e = np.floor(np.log2(np.maximum(np.abs(x), 1e-30)))
    return np.exp2(e - mant_bits)


def assert_rope_close(gpu: np.ndarray, orc: np.ndarray, dtype: int, what: str):
    """RoPE results: the GPU evaluates x*cos - y*sin in fp32, the oracle in
    double; each rounds once to the dtype.  Bound per element: one ulp of the
    dtype at the oracle value, plus the fp32 evaluation error, which is at
    most a few units of 2^-24 of |x| + |y| <= sqrt(2) * |(x', y')| (the
    rotation keeps the pair's magnitude).  The second term only matters where
    the two products nearly cancel."""
    g = W.storage_to_f32(gpu, dtype).astype(np.float64)
    o = W.storage_to_f32(orc, dtype).astype(np.float64)
    both_nan = np.isnan(g) & np.isnan(o)  # canary slots never written
    half = o.shape[-1] // 2
    partner = np.concatenate([o[..., half:], o[..., :half]], axis=-1)
    pairmag = np.sqrt(np.nan_to_num(o) ** 2 + np.nan_to_num(partner) ** 2)
    mant = 7 if dtype == W.BF16 else 23
    allowed = _ulp(o, mant) + 2.0 ** -20 * pairmag
    ok = both_nan | (np.abs(g - o) <= allowed)
    assert ok.all(), (f"{what}: {int((~ok).sum())} elements outside the bound, worst diff "
                      f"{np.nanmax(np.abs(g - o)[~ok])}")


def assert_bits_equal(gpu: np.ndarray, orc: np.ndarray, what: str):
    a = gpu.view(np.uint16 if gpu.dtype == np.uint16 else np.uint32)
    b = orc.view(np.uint16 if orc.dtype == np.uint16 else np.uint32)
    assert np.array_equal(a, b), f"{what}: {int((a != b).sum())} elements differ"


def assert_out_close(gpu_storage: np.ndarray, orc_out: np.ndarray, dtype: int, what: str):
    g = W.storage_to_f32(gpu_storage, dtype).astype(np.float64)
    assert g.shape == orc_out.shape, (what, g.shape, orc_out.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite GPU output"
    err = np.abs(g - orc_out)
    mx, mean = OUT_TOL[dtype]
    assert err.max(initial=0) <= mx, f"{what}: max abs err {err.max()} > {mx}"
    if err.size:
        assert err.mean() <= mean, f"{what}: mean abs err {err.mean()} > {mean}"


def assert_lse_close(gpu: np.ndarray, orc: np.ndarray, dtype: int, what: str):
    ninf = np.isneginf(orc)
    assert np.array_equal(np.isneginf(gpu), ninf), f"{what}: empty-set rows disagree"
    fin = ~ninf
    if fin.any():
        err = np.abs(gpu[fin].astype(np.float64) - orc[fin])
        assert err.max() <= LSE_TOL[dtype], f"{what}: lse err {err.max()}"


def compare_scenario(sc, gpu, orc, rows_per_pass=None):
    """gpu = runner.run_scenario(sc) output; orc = oracle.run_scenario output."""
    gk, gv, gfrozen, gres, untouched_ok = gpu
    ok_, ov, ofrozen, ores = orc
    dt = sc.desc.dtype
    assert untouched_ok, "a page outside the working sets was written"
    assert np.array_equal(gfrozen, ofrozen), f"frozen_len {gfrozen} vs {ofrozen}"
    assert_rope_close(gk, ok_, dt, "K pool")
    assert_bits_equal(gv, ov, "V pool")
    for i, (g, o) in enumerate(zip(gres, ores)):
        tag = f"{sc.name} pass {i}"
        assert g["status"] == o["status"], f"{tag}: status {g['status']} vs {o['status']}"
        assert_rope_close(g["q_rot"], o["q_rot"], dt, tag + " q_rot")
        rows = None if rows_per_pass is None else rows_per_pass[i]
        sel = np.arange(o["out"].shape[0]) if rows is None else np.asarray(rows)
        assert_out_close(g["out_all"][sel], o["out"][sel], dt, tag + " out")
        assert_lse_close(g["lse_all"][sel], o["lse"][sel], dt, tag + " lse")
        ro = o["readout_rows"]
        assert g["out_readout"].shape[0] == ro.shape[0]
        # readout rows are the same rows' outputs, bit for bit
        assert_bits_equal(g["out_readout"], g["out_all"][ro], tag + " readout gather")
        assert np.array_equal(g["lse_readout"].view(np.uint32),
                              g["lse_all"][ro].view(np.uint32)), tag + " readout lse"
        ro_sel = np.isin(ro, sel)
        assert_out_close(g["out_readout"][ro_sel], o["out"][ro[ro_sel]], dt, tag + " readout")
