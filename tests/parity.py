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


def assert_rope_close(gpu: np.ndarray, orc: np.ndarray, dtype: int, what: str):
    if dtype == W.BF16:
        d = np.abs(bf16_ord(gpu) - bf16_ord(orc))
        assert d.max(initial=0) <= 1, f"{what}: {int(d.max())} bf16 ulps apart"
    else:
        g = gpu.astype(np.float64)
        o = orc.astype(np.float64)
        both_nan = np.isnan(g) & np.isnan(o)
        ok = both_nan | (np.abs(g - o) <= 2e-6 + 2e-6 * np.abs(o))
        assert ok.all(), f"{what}: max diff {np.nanmax(np.abs(g - o))}"


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
