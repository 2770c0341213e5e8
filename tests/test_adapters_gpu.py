"""Per-lane adapters (pie_fwd_adapter_plan / pie_fwd_adapter_apply; Pie "The
forward pass", Adapters) against the oracle on the same seeded inputs.

Tolerance, from the arithmetic: the GPU forms A_a x on the tensor cores
(exact bf16 products, fp32 sums over d_in in 64-column chunks and up to 8
ranges), B_a t, y + c_a B_a t and the IA3 product in fp32, and rounds y' to
bf16 once.  With M = the oracle run on absolute values (every term of y'
taken positive), the fp32 part is bounded by about (d_in / 64 + 8 + r + 4)
* 2^-23 * M, well under 1e-4 * M for the shapes here, and the final rounding
by 2^-9 of the result; each element must satisfy
    |got - want| <= 2^-8 |want| + 1e-4 M.
Rows of lanes without an adapter must come back bit for bit."""
import numpy as np
import pytest

import oracle.adapters as OA
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from programmable_paged_kv_gb300 import build
    build()


def _dev(a):
    from programmable_paged_kv_gb300 import runner
    return None if a is None else runner.to_device(a, W.BF16)


def _run(site, max_rank=None, d_out_override=None):
    import torch
    from programmable_paged_kv_gb300 import AdapterPlan, runner
    x, y = _dev(site.x), _dev(site.y)
    la, lb, s = _dev(site.lora_a), _dev(site.lora_b), _dev(site.ia3)
    sc = torch.from_numpy(site.scale).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    mr = site.rank if max_rank is None else max_rank
    plan = AdapterPlan(site.row_indptr, site.adapter_of_lane, len(site.scale), mr)
    plan.apply(x, y, la, lb, sc, s, status=st)
    torch.cuda.synchronize()
    out = runner.to_host(y, W.BF16)
    plan.close()
    return out, int(st.item()), plan.num_tiles


def _f64(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def _expect(site):
    x, y = _f64(site.x), _f64(site.y)
    n_ad = len(site.scale)
    if site.rank > 0:
        A, B = _f64(site.lora_a), _f64(site.lora_b)
        sc = site.scale.astype(np.float64)
    else:
        A = np.zeros((n_ad, 1, x.shape[1]))
        B = np.zeros((n_ad, y.shape[1], 1))
        sc = np.zeros(n_ad)
    s = None if site.ia3 is None else _f64(site.ia3)
    args = (site.row_indptr, site.adapter_of_lane)
    want = OA.apply_adapters(x, y, *args, A, B, sc, s)
    mag = OA.apply_adapters(np.abs(x), np.abs(y), *args, np.abs(A), np.abs(B), np.abs(sc),
                            None if s is None else np.abs(s))
    return want, mag


def _untouched_rows(site):
    keep = np.zeros(site.y.shape[0], bool)
    for l, a in enumerate(site.adapter_of_lane):
        if a < 0:
            keep[site.row_indptr[l]:site.row_indptr[l + 1]] = True
    return keep


def _check(site, got_bits, status):
    assert status == 0
    keep = _untouched_rows(site)
    assert np.array_equal(got_bits[keep], site.y[keep]), "a row without an adapter changed"
    got = _f64(got_bits)
    want, mag = _expect(site)
    err = np.abs(got - want)
    tol = 2.0 ** -8 * np.abs(want) + 1e-4 * mag
    bad = err > tol
    if bad.any():
        r, c = np.argwhere(bad)[0]
        raise AssertionError(f"{int(bad.sum())} elements outside tolerance; first at row {r} col {c}: "
                             f"got {got[r, c]} want {want[r, c]} tol {tol[r, c]}")
    # the bound is loose per element; on average the error sits near the bf16 rounding
    rel = err[~keep] / np.maximum(np.abs(want[~keep]), 1e-3)
    assert rel.size == 0 or float(np.median(rel)) < 2.0 ** -9


CASES = {
    # decode batch shape: one row per lane, q site of a 32 x 128-head model
    "decode_64x1_r16": dict(rows=[1] * 64, d_in=4096, d_out=4096, rank=16, n_adapters=16),
    # ragged lanes: empty, 1, 15, 16, 17 rows, tile edges at 127/128/129, a lane of 3 tiles
    "ragged_r16": dict(rows=[0, 1, 15, 16, 17, 33, 127, 128, 129, 300, 2, 64], d_in=320,
                       d_out=512, rank=16, n_adapters=5, none_every=5),
    "ragged_r8": dict(rows=[3, 130, 16, 1, 40], d_in=256, d_out=768, rank=8, n_adapters=3,
                      none_every=4),
    "ragged_r32": dict(rows=[3, 130, 16, 1, 40], d_in=256, d_out=768, rank=32, n_adapters=3,
                       none_every=4),
    "ragged_r64": dict(rows=[3, 130, 16, 1, 40], d_in=256, d_out=768, rank=64, n_adapters=3,
                       none_every=4),
    "no_ia3_r16": dict(rows=[5, 64, 1, 20], d_in=512, d_out=256, rank=16, n_adapters=2,
                       ia3=False, none_every=0),
    "ia3_only": dict(rows=[5, 64, 1, 20, 7], d_in=128, d_out=512, rank=0, n_adapters=3,
                     none_every=3),
    # 13 chunks of d_in over few tiles: uneven d_in ranges (2 chunks each, one short)
    "uneven_splits": dict(rows=[5, 5, 5], d_in=64 * 13, d_out=256, rank=16, n_adapters=2,
                          none_every=0),
    # a single chunk of d_in, one range
    "one_chunk": dict(rows=[1, 2, 128], d_in=64, d_out=256, rank=16, n_adapters=2,
                      none_every=0),
    # guidance-pair prefill shape: 64 lanes x 64 rows, q site
    "prefill_64x64_r16": dict(rows=[64] * 64, d_in=4096, d_out=4096, rank=16, n_adapters=16),
    # few rows per adapter (the grouped path, a cluster per adapter): eighths
    # of d_in of 5 vectors, 32-column eighths of d_out, every rank, no IA3,
    # an adapter with exactly 16 rows; 17 rows on one adapter takes the tiles
    "grouped_r8": dict(rows=[1, 2, 1, 3, 1, 4, 2], d_in=320, d_out=512, rank=8, n_adapters=3,
                       none_every=4),
    "grouped_r32": dict(rows=[1] * 40, d_in=1024, d_out=768, rank=32, n_adapters=8,
                        none_every=6),
    "grouped_r64": dict(rows=[2, 1, 3, 2, 1, 1], d_in=256, d_out=256, rank=64, n_adapters=2,
                        none_every=0),
    "grouped_no_ia3": dict(rows=[1] * 10, d_in=512, d_out=1024, rank=16, n_adapters=4,
                           ia3=False, none_every=0),
    "grouped_16_rows": dict(rows=[15, 1], d_in=512, d_out=512, rank=16, n_adapters=1,
                            none_every=0),
    "grouped_4_rows": dict(rows=[1] * 8, d_in=2048, d_out=1536, rank=16, n_adapters=8,
                           none_every=0),
    "tiles_17_rows": dict(rows=[16, 1], d_in=512, d_out=512, rank=16, n_adapters=1,
                          none_every=0),
}


@pytest.mark.parametrize("name", list(CASES))
def test_adapters_match_the_oracle(name):
    c = dict(CASES[name])
    rows = c.pop("rows")
    site = W.adapter_site(3, rows, **c)
    got, status, _ = _run(site)
    _check(site, got, status)


def test_a_plan_serves_several_sites_and_a_smaller_rank():
    # one plan (max_rank 32) applied at a q-shaped and at a k-shaped site
    rows = [1, 17, 64, 3]
    q_site = W.adapter_site(5, rows, n_adapters=4, d_in=1024, d_out=1024, rank=16, none_every=3)
    k_site = W.adapter_site(6, rows, n_adapters=4, d_in=1024, d_out=256, rank=32, none_every=3)
    k_site.adapter_of_lane = q_site.adapter_of_lane.copy()
    import torch
    from programmable_paged_kv_gb300 import AdapterPlan, runner
    plan = AdapterPlan(q_site.row_indptr, q_site.adapter_of_lane, 4, 32)
    outs = []
    for site in (q_site, k_site):
        x, y = _dev(site.x), _dev(site.y)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        plan.apply(x, y, _dev(site.lora_a), _dev(site.lora_b),
                   torch.from_numpy(site.scale).cuda(), _dev(site.ia3), status=st)
        torch.cuda.synchronize()
        outs.append((runner.to_host(y, W.BF16), int(st.item())))
    plan.close()
    for site, (got, status) in zip((q_site, k_site), outs):
        _check(site, got, status)


def test_lanes_without_adapters_launch_nothing_and_keep_y():
    site = W.adapter_site(7, [4, 9, 1], n_adapters=2, d_in=128, d_out=256, rank=16,
                          none_every=1)
    got, status, tiles = _run(site)
    assert tiles == 0 and status == 0
    assert np.array_equal(got, site.y)


def test_results_are_deterministic():
    site = W.adapter_site(8, [64, 1, 130], n_adapters=2, d_in=1024, d_out=512, rank=16,
                          none_every=0)
    a, _, _ = _run(site)
    b, _, _ = _run(site)
    assert np.array_equal(a, b)
