"""Pins of the CPU oracle against what the Pie pages and plain mathematics fix.

Each test checks the oracle against something other than itself: a worked
example printed in the pages (tests/golden/), a closed form, a library
routine (torch's bf16 rounding, numpy complex exponentials, scipy's softmax),
an invariant the pages state (folding() is causal; prefix + continuation
equals one monolithic pass; a sliding-window mask equals attention over the
truncated working set; masking never touches the cache) or brute force on
tiny inputs.  The cases are chosen so that a dropped term, a flipped sign, a
wrong index or swapped K/V operands fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle as O
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers
def one_lane_pass(desc, kv_len, pages, positions, slots, q, k, v, fold=W.FOLD_NONE,
                  mask_rows=None, readout=None, fold_count=0):
    N = len(positions)
    p = W.Pass(row_indptr=np.array([0, N], np.int32),
               positions=np.asarray(positions, np.int32), slots=np.asarray(slots, np.int32),
               kv_len=np.array([kv_len], np.int32), page_indptr=np.array([0, len(pages)], np.int32),
               page_ids=np.asarray(pages, np.int32), fold_mode=np.array([fold], np.int32),
               fold_count=np.array([fold_count], np.int32),
               q=np.ascontiguousarray(q), k=np.ascontiguousarray(k), v=np.ascontiguousarray(v),
               readout=None if readout is None else np.asarray(readout, np.int32))
    if mask_rows is not None:
        p.mask_word_indptr, p.mask_words = W.mask_from_visible(mask_rows)
    return p


def f32_desc(Hq=1, Hkv=1, d=4, P=8):
    return W.Desc(Hq, Hkv, d, P, W.F32)


def pools(desc, npages, fill=np.nan):
    shape = (npages, desc.num_kv_heads, desc.page_size, desc.head_dim)
    return np.full(shape, fill, np.float32), np.full(shape, fill, np.float32)


def preload(desc, kp, vp, pages, Kc, Vc):
    """Write cached K/V [T, Hkv, d] for slots 0..T-1 of a lane (no rotation)."""
    P = desc.page_size
    for s in range(Kc.shape[0]):
        kp[pages[s // P], :, s % P, :] = Kc[s]
        vp[pages[s // P], :, s % P, :] = Vc[s]


def attend_cached(desc, Kc, Vc, q, visible=None, pages=None, npages=None, fold=W.FOLD_NONE):
    """One row at position 0 (no rotation) attending over cached slots 0..T-1.

    The row itself writes its (zero) K/V into slot T, which is excluded by
    kv_len = T unless visible says otherwise."""
    T = Kc.shape[0]
    P = desc.page_size
    need = T // P + 1
    pages = list(range(need)) if pages is None else pages
    npages = npages or max(pages) + 1
    kp, vp = pools(desc, npages)
    preload(desc, kp, vp, pages, Kc, Vc)
    Hq, Hkv, d = desc.num_q_heads, desc.num_kv_heads, desc.head_dim
    zero = np.zeros((1, Hkv, d), np.float32)
    p = one_lane_pass(desc, T, pages, [0], [T], q.reshape(1, Hq, d).astype(np.float32),
                      zero, zero, fold=fold,
                      mask_rows=None if visible is None else [np.asarray(visible, bool)])
    frozen = np.array([T], np.int32)
    r = O.run_pass(desc, p, kp, vp, frozen)
    assert r["err"] == O.OK
    return r


# ---------------------------------------------------------------- dtype
def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    xs = np.concatenate([
        rng.standard_normal(2000).astype(np.float32),
        (rng.standard_normal(500) * 1e-38).astype(np.float32),   # subnormal range
        (rng.standard_normal(500) * 1e37).astype(np.float32),
        np.array([1.0 + 2**-8, 1.0 + 3 * 2**-8, -1.0 - 2**-8, 3.0e38, -3.39e38, 0.0, -0.0,
                  2**-133, 2**-134, 1.5 * 2**-133], np.float32),  # ties and edges
    ])
    want = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([O.round_bf16(float(x)) for x in xs], np.uint16)
    np.testing.assert_array_equal(got, want)


# ---------------------------------------------------------------- RoPE
def test_rope_position_zero_is_identity():
    desc = W.Desc(1, 1, 64, 16, W.F32)
    x = np.random.default_rng(0).standard_normal(64)
    np.testing.assert_array_equal(O.rope(desc, x, 0), x)


def test_rope_unit_vectors_closed_form():
    """e_0 turns by angle pos (frequency base^0 = 1) towards e_{d/2}; e_{d/4}
    turns by pos * base^(-1/2) = pos / 100 at base 10000."""
    d = 64
    desc = W.Desc(1, 1, d, 16, W.F32, rope_base=10000.0)
    for pos in (1, 7, 1000):
        e0 = np.zeros(d)
        e0[0] = 1.0
        y = O.rope(desc, e0, pos)
        assert y[0] == pytest.approx(math.cos(pos), abs=1e-12)
        assert y[d // 2] == pytest.approx(math.sin(pos), abs=1e-12)
        assert np.count_nonzero(y) == 2
        eq = np.zeros(d)
        eq[d // 4] = 1.0
        y = O.rope(desc, eq, pos)
        ang = float(np.float32(pos) * np.float32(0.01))
        assert y[d // 4] == pytest.approx(math.cos(ang), abs=1e-6)
        assert y[d // 4 + d // 2] == pytest.approx(math.sin(ang), abs=1e-6)
        # the partner component turns the other way: e_{d/2} -> -sin on e_0
        eh = np.zeros(d)
        eh[d // 2] = 1.0
        y = O.rope(desc, eh, pos)
        assert y[0] == pytest.approx(-math.sin(pos), abs=1e-12)
        assert y[d // 2] == pytest.approx(math.cos(pos), abs=1e-12)


def test_rope_is_complex_rotation():
    """Rotate-half RoPE equals multiplying z_i = x_i + i x_{i+d/2} by
    exp(i * theta_i) (numpy's complex exponential)."""
    d = 128
    desc = W.Desc(1, 1, d, 16, W.F32)
    rng = np.random.default_rng(2)
    x = rng.standard_normal(d)
    i = np.arange(d // 2)
    for pos in (3, 511, 32767):
        freq = np.array([np.float32(10000.0 ** (-2.0 * k / d)) for k in i], np.float32)
        theta = (np.float32(pos) * freq).astype(np.float64)
        z = (x[: d // 2] + 1j * x[d // 2:]) * np.exp(1j * theta)
        y = O.rope(desc, x, pos)
        np.testing.assert_allclose(y[: d // 2], z.real, rtol=0, atol=1e-12)
        np.testing.assert_allclose(y[d // 2:], z.imag, rtol=0, atol=1e-12)


def test_rope_norm_and_relative_position():
    d = 64
    desc = W.Desc(1, 1, d, 16, W.F32)
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    for p, s, delta in ((5, 2, 100), (40, 39, 7), (17, 0, 1000)):
        assert np.linalg.norm(O.rope(desc, q, p)) == pytest.approx(np.linalg.norm(q), rel=1e-12)
        a = O.rope(desc, q, p) @ O.rope(desc, k, s)
        b = O.rope(desc, q, p + delta) @ O.rope(desc, k, s + delta)
        # fp32 angles: the invariance holds up to the angle rounding
        assert a == pytest.approx(b, abs=2e-3 * np.linalg.norm(q) * np.linalg.norm(k))


# ---------------------------------------------------------------- Eq. (1), Eq. (2)
def test_kv_bytes_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "kv_bytes_eq1.json")))
    per_tok = O.kv_bytes(g["layers"], g["kv_heads"], g["head_dim"], 1, g["elem_bytes"])
    assert per_tok == g["bytes_per_token"]
    assert O.kv_bytes(g["layers"], g["kv_heads"], g["head_dim"], g["tokens"],
                      g["elem_bytes"]) == g["bytes_total"]


def test_page_waste_cases():
    g = json.load(open(os.path.join(GOLDEN, "page_waste_eq2.json")))
    for c in g["cases"]:
        assert O.page_waste(c["T"], c["P"]) == c["W"]
    for P in (8, 16, 32):
        for T in range(0, 200):
            assert 0 <= O.page_waste(T, P) < P


def test_scatter_writes_exactly_eq1_bytes_and_leaves_eq2_waste():
    """After the tiny folding() scenario (48 tokens), the pools hold exactly
    M_KV(L=1, Hkv, d, T=48, b=4) bytes of written data; after its 40-row
    prefill alone, the unwritten slots of the lane's ceil(40/16) pages are
    W(40, 16) per head."""
    sc = W.tiny(0)
    d = sc.desc
    k, v, frozen, _ = O.run_scenario(sc)
    written = (~np.isnan(k)).sum() + (~np.isnan(v)).sum()
    assert written * 4 == O.kv_bytes(1, d.num_kv_heads, d.head_dim, 48, 4)
    assert frozen[0] == 48
    k = sc.k_init.copy()
    v = sc.v_init.copy()
    fr = sc.frozen_len0.copy()
    p = sc.passes[0]
    r = O.run_pass(d, p, k, v, fr, page_ids=sc.compact_page_ids(p.page_ids))
    assert r["err"] == O.OK
    lane_pages = sc.compact_page_ids(p.page_ids)[: -(-40 // d.page_size)]
    unwritten_slots = np.isnan(k[lane_pages][:, 0, :, 0]).sum()
    assert unwritten_slots == O.page_waste(40, d.page_size)


# ---------------------------------------------------------------- attention closed forms
def test_single_visible_slot_returns_its_value():
    desc = f32_desc(d=4)
    rng = np.random.default_rng(4)
    Kc = rng.standard_normal((6, 1, 4)).astype(np.float32)
    Vc = rng.standard_normal((6, 1, 4)).astype(np.float32)
    q = rng.standard_normal(4).astype(np.float32)
    for s in range(6):
        vis = np.zeros(6, bool)
        vis[s] = True
        r = attend_cached(desc, Kc, Vc, q, visible=vis)
        np.testing.assert_array_equal(r["out"][0, 0], Vc[s, 0].astype(np.float64))
        z = float(q.astype(np.float64) @ Kc[s, 0].astype(np.float64)) / 2.0
        assert r["lse"][0, 0] == pytest.approx(z, rel=1e-15, abs=1e-15)


def test_two_slots_closed_form_and_scale():
    """q.k1 = 8, q.k2 = 0 with d = 16: weights are sigmoid(+-8/sqrt(16))."""
    d = 16
    desc = f32_desc(d=d)
    q = np.zeros(d, np.float32)
    q[0] = 2.0
    Kc = np.zeros((2, 1, d), np.float32)
    Kc[0, 0, 0] = 4.0           # q.k1 = 8
    Vc = np.zeros((2, 1, d), np.float32)
    Vc[0, 0, 1] = 1.0
    Vc[1, 0, 2] = 1.0
    r = attend_cached(desc, Kc, Vc, q)
    w1 = 1.0 / (1.0 + math.exp(-2.0))  # 8 / sqrt(16) = 2
    assert r["out"][0, 0, 1] == pytest.approx(w1, rel=1e-14)
    assert r["out"][0, 0, 2] == pytest.approx(1 - w1, rel=1e-14)
    assert r["lse"][0, 0] == pytest.approx(math.log(math.exp(2.0) + 1.0), rel=1e-14)


def test_zero_query_gives_uniform_mean_and_log_count():
    desc = f32_desc(d=8, P=4)
    rng = np.random.default_rng(5)
    T = 11
    Kc = rng.standard_normal((T, 1, 8)).astype(np.float32)
    Vc = np.zeros((T, 1, 8), np.float32)
    for s in range(T):
        Vc[s, 0, s % 8] = s + 1.0
    r = attend_cached(desc, Kc, Vc, np.zeros(8, np.float32))
    assert r["lse"][0, 0] == pytest.approx(math.log(T), rel=1e-15)
    np.testing.assert_allclose(r["out"][0, 0], Vc[:, 0].astype(np.float64).mean(0), rtol=1e-14)


def test_identical_keys_give_mean_of_visible_values():
    desc = f32_desc(d=4)
    rng = np.random.default_rng(6)
    Kc = np.repeat(rng.standard_normal((1, 1, 4)).astype(np.float32), 7, 0)
    Vc = rng.standard_normal((7, 1, 4)).astype(np.float32)
    vis = np.array([1, 0, 1, 1, 0, 0, 1], bool)
    r = attend_cached(desc, Kc, Vc, rng.standard_normal(4).astype(np.float32), visible=vis)
    np.testing.assert_allclose(r["out"][0, 0], Vc[vis, 0].astype(np.float64).mean(0),
                               rtol=1e-13, atol=1e-15)


def test_gqa_heads_read_their_group():
    """Hq=4, Hkv=2: q heads 0,1 read kv head 0, heads 2,3 read kv head 1."""
    desc = f32_desc(Hq=4, Hkv=2, d=4)
    Kc = np.zeros((3, 2, 4), np.float32)
    Vc = np.zeros((3, 2, 4), np.float32)
    Vc[:, 0, :] = 1.0
    Vc[:, 1, :] = 2.0
    r = attend_cached(desc, Kc, Vc, np.ones((4, 4), np.float32))
    np.testing.assert_array_equal(r["out"][0, :, 0], [1.0, 1.0, 2.0, 2.0])


def test_default_visibility_is_causal_in_slot_space():
    """One-hot values and a zero query expose the visible set of every row of
    a 10-row prefill: row at slot s sees exactly slots 0..s."""
    d, T = 16, 10
    desc = f32_desc(d=d, P=4)
    pages = [3, 0, 2]
    kp, vp = pools(desc, 4)
    q = np.zeros((T, 1, d), np.float32)
    k = np.random.default_rng(7).standard_normal((T, 1, d)).astype(np.float32)
    v = np.zeros((T, 1, d), np.float32)
    for s in range(T):
        v[s, 0, s] = 1.0
    p = one_lane_pass(desc, T, pages, list(range(T)), list(range(T)), q, k, v, fold=W.FOLD_ALL)
    r = O.run_pass(desc, p, kp, vp, np.zeros(1, np.int32))
    for s in range(T):
        want = np.zeros(d)
        want[: s + 1] = 1.0 / (s + 1)
        np.testing.assert_allclose(r["out"][s, 0], want, rtol=1e-15)


def test_mask_bits_lsb_first_and_kv_len_bound():
    """Bit (s & 31) of word s >> 5 selects slot s; bits at or past kv_len are
    ignored (here kv_len = 37 with bits 37..63 set)."""
    d, T = 64, 37
    desc = f32_desc(d=d, P=16)
    Kc = np.zeros((T, 1, d), np.float32)
    Vc = np.zeros((T, 1, d), np.float32)
    for s in range(T):
        Vc[s, 0, s] = 1.0
    vis_set = [0, 5, 31, 32, 36]
    words = np.zeros(2, np.uint32)
    for s in vis_set + list(range(37, 64)):
        words[s >> 5] |= np.uint32(1 << (s & 31))
    pages = [0, 1, 2]
    kp, vp = pools(desc, 3)
    preload(desc, kp, vp, pages, Kc, Vc)
    z = np.zeros((1, 1, d), np.float32)
    p = one_lane_pass(desc, T, pages, [0], [T], z, z, z)
    p.mask_word_indptr = np.array([0, 2], np.int64)
    p.mask_words = words
    r = O.run_pass(desc, p, kp, vp, np.array([T], np.int32))
    want = np.zeros(d)
    want[vis_set] = 1.0 / len(vis_set)
    np.testing.assert_allclose(r["out"][0, 0], want, rtol=1e-15)


def test_empty_visible_set():
    desc = f32_desc(d=4)
    Kc = np.ones((4, 1, 4), np.float32)
    r = attend_cached(desc, Kc, Kc, np.ones(4, np.float32), visible=np.zeros(4, bool))
    np.testing.assert_array_equal(r["out"][0, 0], np.zeros(4))
    assert r["lse"][0, 0] == -np.inf


def test_brute_force_all_masks_against_scipy_softmax():
    """d = 4, kv_len = 8: every one of the 256 masks of one row against a
    dense restatement using scipy.special.softmax / logsumexp."""
    sp = pytest.importorskip("scipy.special")
    desc = f32_desc(d=4, P=4)
    rng = np.random.default_rng(8)
    T = 8
    Kc = rng.standard_normal((T, 1, 4)).astype(np.float32)
    Vc = rng.standard_normal((T, 1, 4)).astype(np.float32)
    q = rng.standard_normal(4).astype(np.float32)
    z = (Kc[:, 0].astype(np.float64) @ q.astype(np.float64)) / 2.0
    for bits in range(1, 256):
        vis = np.array([(bits >> s) & 1 for s in range(T)], bool)
        r = attend_cached(desc, Kc, Vc, q, visible=vis, pages=[1, 0, 2], npages=3)
        w = sp.softmax(z[vis])
        np.testing.assert_allclose(r["out"][0, 0], w @ Vc[vis, 0].astype(np.float64),
                                   rtol=1e-12, atol=1e-14)
        assert r["lse"][0, 0] == pytest.approx(sp.logsumexp(z[vis]), rel=1e-13)


# ---------------------------------------------------------------- invariants from the pages
def test_folding_equals_explicit_causal_mask():
    """folding() appends causally; the same pass with explicit causal mask
    words gives bit-identical outputs (Pie: State geometry; Attention masks)."""
    for name in ("tiny", "guidance_pairs", "spec_verify"):
        sc = W.small(name, 3)
        _, _, _, base = O.run_scenario(sc)
        for i, p in enumerate(sc.passes):
            vis = []
            for l in range(p.num_lanes):
                for r in range(p.row_indptr[l], p.row_indptr[l + 1]):
                    s = np.arange(p.kv_len[l])
                    vis.append(s <= p.slots[r])
            p.mask_word_indptr, p.mask_words = W.mask_from_visible(vis)
        _, _, _, masked = O.run_scenario(sc)
        for a, b in zip(base, masked):
            np.testing.assert_array_equal(a["out"], b["out"])
            np.testing.assert_array_equal(a["lse"], b["lse"])


def test_prefix_then_continuation_equals_monolithic_pass():
    """40-row prefix + 8 single-row continuations over the retained cache ==
    one 48-row pass (Pie review section 4's equivalence check)."""
    sc = W.tiny(5)
    d = sc.desc
    k_s, v_s, fr_s, split = O.run_scenario(sc)
    split_out = np.concatenate([r["out"] for r in split], 0)
    split_qrot = np.concatenate([r["q_rot"] for r in split], 0)
    P0 = sc.passes[0]
    T = 48
    mono = W.Pass(row_indptr=np.array([0, T], np.int32), positions=np.arange(T, dtype=np.int32),
                  slots=np.arange(T, dtype=np.int32), kv_len=np.array([T], np.int32),
                  page_indptr=P0.page_indptr, page_ids=P0.page_ids,
                  fold_mode=np.array([W.FOLD_ALL], np.int32), fold_count=np.zeros(1, np.int32),
                  q=np.concatenate([p.q for p in sc.passes]),
                  k=np.concatenate([p.k for p in sc.passes]),
                  v=np.concatenate([p.v for p in sc.passes]))
    k_m, v_m = sc.k_init.copy(), sc.v_init.copy()
    fr_m = sc.frozen_len0.copy()
    r = O.run_pass(d, mono, k_m, v_m, fr_m, page_ids=sc.compact_page_ids(mono.page_ids))
    np.testing.assert_array_equal(r["out"], split_out)
    np.testing.assert_array_equal(r["q_rot"], split_qrot)
    np.testing.assert_array_equal(k_m.view(np.uint32), k_s.view(np.uint32))
    np.testing.assert_array_equal(v_m.view(np.uint32), v_s.view(np.uint32))
    assert fr_m[0] == fr_s[0] == T


def test_sliding_window_equals_truncated_working_set():
    """Sinks + window mask == causal attention over a working set holding only
    the sink and window slots (copied with their already-rotated K), queried
    at the row's original position (Pie: Attention masks)."""
    sc = W.masked_long(4, "window", lanes=1, kv=300, rows=6, sinks=4, window=50,
                       desc=W.Desc(4, 2, 64, 16, W.F32))
    d = sc.desc
    k, v, fr, (res,) = O.run_scenario(sc)
    p = sc.passes[0]
    cpages = sc.compact_page_ids(p.page_ids)
    P = d.page_size
    for i in range(p.num_rows):
        pos = int(p.positions[i])
        keep = [s for s in range(4)] + list(range(pos - 49, pos))  # excluding own slot
        Tn = len(keep) + 1
        npg = -(-Tn // P)
        kt, vt = pools(d, npg)
        for j, s in enumerate(keep):
            kt[j // P, :, j % P] = k[cpages[s // P], :, s % P]
            vt[j // P, :, j % P] = v[cpages[s // P], :, s % P]
        t = one_lane_pass(d, Tn, list(range(npg)), [pos], [Tn - 1], p.q[i:i + 1], p.k[i:i + 1],
                          p.v[i:i + 1], fold=W.FOLD_ALL)
        r = O.run_pass(d, t, kt, vt, np.array([Tn - 1], np.int32))
        np.testing.assert_array_equal(r["out"][0], res["out"][i])
        np.testing.assert_array_equal(r["lse"][0], res["lse"][i])


def test_masking_never_modifies_the_cache():
    """Pools after a pass are bit-identical whatever the mask and whether or
    not attention ran (Pie review section 3: masking is not recompute)."""
    sc = W.small("masked_tova", 2)
    d = sc.desc
    p = sc.passes[0]
    cp = sc.compact_page_ids(p.page_ids)
    outs = []
    for use_mask, rows in ((True, None), (False, None), (True, np.zeros(0, np.int32))):
        k, v, fr = sc.k_init.copy(), sc.v_init.copy(), sc.frozen_len0.copy()
        O.run_pass(d, p, k, v, fr, page_ids=cp, rows=rows, use_mask=use_mask)
        outs.append((k, v))
    for k, v in outs[1:]:
        np.testing.assert_array_equal(k, outs[0][0])
        np.testing.assert_array_equal(v, outs[0][1])


def test_physical_page_permutation_is_invisible():
    sc = W.small("decode_batch", 4)
    d = sc.desc
    _, _, _, (base,) = O.run_scenario(sc)
    U = sc.pool_pages.size
    perm = np.random.default_rng(9).permutation(U)
    k = np.empty_like(sc.k_init)
    v = np.empty_like(sc.v_init)
    k[perm] = sc.k_init
    v[perm] = sc.v_init
    p = sc.passes[0]
    fr = sc.frozen_len0.copy()
    r = O.run_pass(d, p, k, v, fr, page_ids=perm[sc.compact_page_ids(p.page_ids)].astype(np.int32))
    np.testing.assert_array_equal(r["out"], base["out"])


def _lane_subpass(p, l):
    """Lane l of a multi-lane pass as a pass of its own (same pages, rows)."""
    r0, r1 = int(p.row_indptr[l]), int(p.row_indptr[l + 1])
    g0, g1 = int(p.page_indptr[l]), int(p.page_indptr[l + 1])
    sub = W.Pass(row_indptr=np.array([0, r1 - r0], np.int32), positions=p.positions[r0:r1].copy(),
                 slots=p.slots[r0:r1].copy(), kv_len=p.kv_len[l:l + 1].copy(),
                 page_indptr=np.array([0, g1 - g0], np.int32), page_ids=p.page_ids[g0:g1].copy(),
                 fold_mode=p.fold_mode[l:l + 1].copy(), fold_count=p.fold_count[l:l + 1].copy(),
                 q=p.q[r0:r1].copy(), k=p.k[r0:r1].copy(), v=p.v[r0:r1].copy())
    if p.mask_word_indptr is not None:
        w0, w1 = int(p.mask_word_indptr[r0]), int(p.mask_word_indptr[r1])
        sub.mask_word_indptr = (p.mask_word_indptr[r0:r1 + 1] - w0).astype(np.int64)
        sub.mask_words = p.mask_words[w0:w1].copy()
    return sub


@pytest.mark.parametrize("name", ["decode_batch", "guidance_pairs", "masked_tova"])
def test_lanes_are_independent(name):
    """A multi-lane pass equals each lane run alone on its own working set
    (Pie: Lanes -- each lane has its own tokens and its own working set)."""
    sc = W.small(name, 11)
    d = sc.desc
    p = sc.passes[0]
    k, v, fr = sc.k_init.copy(), sc.v_init.copy(), sc.frozen_len0.copy()
    full = O.run_pass(d, p, k, v, fr, page_ids=sc.compact_page_ids(p.page_ids))
    for l in range(p.num_lanes):
        sub = _lane_subpass(p, l)
        k1, v1 = sc.k_init.copy(), sc.v_init.copy()
        fr1 = sc.frozen_len0[l:l + 1].copy()
        r = O.run_pass(d, sub, k1, v1, fr1, page_ids=sc.compact_page_ids(sub.page_ids))
        r0, r1 = p.row_indptr[l], p.row_indptr[l + 1]
        np.testing.assert_array_equal(r["out"], full["out"][r0:r1])
        assert fr1[0] == fr[l]


# ---------------------------------------------------------------- fold, readout, status
def test_verify_fold_from_channel_and_stale_drafts():
    """Speculative verify: fold=0 drafts, accepted count a from the channel
    freezes C+a slots; the follow-up decode overwrites slot C+a and never
    reads the stale drafts past it (Pie: State geometry)."""
    sc = W.small("spec_verify", 6)
    C = sc.frozen_len0.copy()
    k, v, fr, (r1, r2) = O.run_scenario(sc)
    a = sc.passes[0].channel
    assert (a >= 0).all() and (a <= 8).all()
    # after pass 2 (fold=all, one row) the frozen length is C + a + 1
    np.testing.assert_array_equal(fr, C + a + 1)
    assert r1["status"] == 0 and r2["status"] == 0
    np.testing.assert_array_equal(r1["readout_rows"], np.arange(sc.passes[0].num_rows))
    # stale drafts past C+a are invisible to pass 2: poisoning them changes nothing
    p2 = sc.passes[1]
    cp = sc.compact_page_ids(p2.page_ids)
    P = sc.desc.page_size
    k3, v3 = sc.k_init.copy(), sc.v_init.copy()
    fr3 = sc.frozen_len0.copy()
    O.run_pass(sc.desc, sc.passes[0], k3, v3, fr3, page_ids=sc.compact_page_ids(sc.passes[0].page_ids))
    for l in range(p2.num_lanes):
        for s in range(C[l] + a[l] + 1, C[l] + 8):
            k3[cp[p2.page_indptr[l] + s // P], :, s % P] = W.CANARY[W.BF16]
            v3[cp[p2.page_indptr[l] + s // P], :, s % P] = W.CANARY[W.BF16]
    r = O.run_pass(sc.desc, p2, k3, v3, fr3, page_ids=cp)
    np.testing.assert_array_equal(r["out"], r2["out"])


@pytest.mark.parametrize("chan,want,flag", [(9, 3, True), (-1, 0, True), (2, 2, False),
                                            (3, 3, False), (0, 0, False)])
def test_channel_count_is_clamped_and_flagged(chan, want, flag):
    desc = f32_desc(d=4)
    z = np.zeros((3, 1, 4), np.float32)
    p = one_lane_pass(desc, 8, [0], [5, 6, 7], [5, 6, 7], z, z, z, fold=W.FOLD_CHANNEL)
    kp, vp = pools(desc, 1, 0.0)
    fr = np.array([5], np.int32)
    r = O.run_pass(desc, p, kp, vp, fr, channel=np.array([chan], np.int32))
    assert fr[0] == 5 + want
    assert bool(r["status"] & O.ST_FOLD_CLAMP) == flag


def test_fold_modes():
    desc = f32_desc(d=4)
    z = np.zeros((4, 1, 4), np.float32)
    for mode, cnt, want in ((W.FOLD_NONE, 0, 0), (W.FOLD_ALL, 0, 4), (W.FOLD_COUNT, 3, 3)):
        p = one_lane_pass(desc, 6, [0], [2, 3, 4, 5], [2, 3, 4, 5], z, z, z, fold=mode,
                          fold_count=cnt)
        kp, vp = pools(desc, 1, 0.0)
        fr = np.array([2], np.int32)
        r = O.run_pass(desc, p, kp, vp, fr)
        assert r["status"] == 0 and fr[0] == 2 + want


def test_frozen_write_is_skipped_and_flagged():
    desc = f32_desc(d=4)
    q = np.ones((2, 1, 4), np.float32)
    k = np.full((2, 1, 4), 7.0, np.float32)
    p = one_lane_pass(desc, 6, [0], [0, 0], [2, 5], q, k, k)
    kp, vp = pools(desc, 1, 0.0)
    fr = np.array([4], np.int32)
    r = O.run_pass(desc, p, kp, vp, fr)
    assert r["status"] & O.ST_FROZEN_WRITE
    assert (kp[0, 0, 2] == 0).all() and (kp[0, 0, 5] == 7.0).all()


def test_fold_gap_is_flagged():
    desc = f32_desc(d=4)
    z = np.zeros((1, 1, 4), np.float32)
    p = one_lane_pass(desc, 6, [0], [5], [5], z, z, z, fold=W.FOLD_ALL)
    kp, vp = pools(desc, 1, 0.0)
    fr = np.array([3], np.int32)
    r = O.run_pass(desc, p, kp, vp, fr)
    assert r["status"] & O.ST_FOLD_GAP and fr[0] == 4


def test_default_readout_is_last_row_per_nonempty_lane():
    desc = f32_desc(d=4)
    p = one_lane_pass(desc, 0, [0, 1, 2], [], [], np.zeros((0, 1, 4), np.float32),
                      np.zeros((0, 1, 4), np.float32), np.zeros((0, 1, 4), np.float32))
    # three lanes: 2 rows, 0 rows, 3 rows
    p.row_indptr = np.array([0, 2, 2, 5], np.int32)
    p.positions = np.array([0, 1, 0, 1, 2], np.int32)
    p.slots = p.positions.copy()
    p.kv_len = np.array([2, 0, 3], np.int32)
    p.page_indptr = np.array([0, 1, 2, 3], np.int32)
    p.fold_mode = np.zeros(3, np.int32)
    p.fold_count = np.zeros(3, np.int32)
    p.q = np.zeros((5, 1, 4), np.float32)
    p.k = p.v = p.q
    kp, vp = pools(desc, 3, 0.0)
    r = O.run_pass(desc, p, kp, vp, np.zeros(3, np.int32))
    assert r["err"] == O.OK
    np.testing.assert_array_equal(r["readout_rows"], [1, 4])


# ---------------------------------------------------------------- validation
def _valid_pass():
    desc = f32_desc(d=4)
    z = np.zeros((2, 1, 4), np.float32)
    return desc, one_lane_pass(desc, 10, [0, 1], [8, 9], [8, 9], z, z, z, fold=W.FOLD_ALL)


@pytest.mark.parametrize("mutate,code", [
    (lambda p: setattr(p, "row_indptr", np.array([0, 3], np.int32)), O.EINVAL),
    (lambda p: setattr(p, "slots", np.array([8, 16], np.int32)), O.ERANGE),
    (lambda p: setattr(p, "slots", np.array([-1, 9], np.int32)), O.ERANGE),
    (lambda p: setattr(p, "positions", np.array([-2, 9], np.int32)), O.ERANGE),
    (lambda p: setattr(p, "kv_len", np.array([17], np.int32)), O.ERANGE),
    (lambda p: setattr(p, "page_ids", np.array([0, 5], np.int32)), O.ERANGE),
    (lambda p: setattr(p, "slots", np.array([9, 8], np.int32)), O.EINVAL),   # fold needs consecutive
    (lambda p: (setattr(p, "fold_mode", np.array([0], np.int32)),
                setattr(p, "slots", np.array([9, 9], np.int32))), O.EINVAL),  # Eq. (4) duplicate
    (lambda p: setattr(p, "fold_mode", np.array([7], np.int32)), O.EINVAL),
    (lambda p: (setattr(p, "fold_mode", np.array([2], np.int32)),
                setattr(p, "fold_count", np.array([3], np.int32))), O.ERANGE),
    (lambda p: setattr(p, "readout", np.array([2], np.int32)), O.ERANGE),
    (lambda p: (setattr(p, "mask_word_indptr", np.array([0, 1, 1], np.int64)),
                setattr(p, "mask_words", np.ones(1, np.uint32))), O.ERANGE),
])
def test_invalid_metadata_is_rejected(mutate, code):
    desc, p = _valid_pass()
    assert O.validate(desc, p, num_pool_pages=2) == O.OK
    mutate(p)
    assert O.validate(desc, p, num_pool_pages=2) == code
