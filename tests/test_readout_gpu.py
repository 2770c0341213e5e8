"""Readout distribution epilogue on the GPU (pie_fwd_readout_topk) against
the oracle (the review "Pie: Who Should Control the LLM Generation Loop?",
section 7, Eq. (6)-(7)): token ids bit-exact (ties by smaller id), p, Z and
lse within fp32 tolerances, over vocabulary sizes that span one to many
slices with ragged tails, fp32 and bf16 logits (bf16 rows are full of ties),
masked (-inf) tokens and degenerate rows."""
import numpy as np
import pytest

import oracle.readout as RO
import workloads as W

pytestmark = pytest.mark.gpu

# p and lse in fp32 on the GPU, float64 in the oracle: the exponent argument
# x - lse carries an fp32 rounding of |x - lse| * 2^-24 (|x - lse| < 64 here),
# the slice normalisers a few ulp each
P_RTOL, P_ATOL = 2e-5, 1e-30
Z_ATOL = 2e-5
LSE_RTOL = 2e-6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from programmable_paged_kv_gb300 import build
    build()


def _run(logits_np, k, dtype="f32", ld=None):
    import torch
    from programmable_paged_kv_gb300 import readout_topk
    R, V = logits_np.shape
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    ld = ld or V
    buf = torch.full((R, ld), -1.0, dtype=torch.float32)
    buf[:, :V] = torch.from_numpy(logits_np.astype(np.float32))
    dev = buf.to(tdt).cuda()
    view = dev[:, :V]
    ids = torch.empty((R, k), dtype=torch.int32, device="cuda")
    probs = torch.empty((R, k), dtype=torch.float32, device="cuda")
    z = torch.empty(R, dtype=torch.float32, device="cuda")
    lse = torch.empty(R, dtype=torch.float32, device="cuda")
    readout_topk(view, k, ids, probs, z, lse)
    torch.cuda.synchronize()
    # what the kernel saw (bf16 logits are rounded before both sides use them)
    seen = view.float().cpu().numpy()
    return seen, ids.cpu().numpy(), probs.cpu().numpy(), z.cpu().numpy(), lse.cpu().numpy()


def _check(seen, k, ids, probs, z, lse):
    e_ids, e_probs, e_z, e_lse = RO.readout_topk(seen, k)
    np.testing.assert_array_equal(ids, e_ids)
    np.testing.assert_allclose(probs, e_probs, rtol=P_RTOL, atol=P_ATOL)
    np.testing.assert_allclose(z, e_z, rtol=0, atol=Z_ATOL)
    np.testing.assert_allclose(lse, e_lse, rtol=LSE_RTOL, atol=1e-6)


CASES = {
    # name: (rows, vocab, k, dtype, ld or None, spikes)
    "full_vocab_f32": (6, 128256, 256, "f32", None, 8),
    "full_vocab_bf16_ties": (5, 128256, 256, "bf16", None, 8),
    "one_short_slice": (3, 300, 256, "f32", None, 2),
    "k_equals_vocab": (2, 100, 100, "f32", None, 0),
    "ragged_tail_padded_rows": (3, 3 * 8192 + 17, 200, "f32", 3 * 8192 + 20, 4),
    "ragged_tail_bf16": (3, 2 * 8192 + 5, 64, "bf16", 2 * 8192 + 8, 4),
    "largest_vocab": (2, 262144, 256, "bf16", None, 8),
    "argmax_k1": (4, 4000, 1, "bf16", None, 1),
    "many_rows": (300, 1000, 32, "f32", None, 3),
}


@pytest.mark.parametrize("name", list(CASES))
def test_readout_topk_matches_oracle(name):
    R, V, k, dt, ld, spikes = CASES[name]
    logits = W.readout_logits(11, R, V, spikes=spikes)
    seen, ids, probs, z, lse = _run(logits, k, dt, ld)
    _check(seen, k, ids, probs, z, lse)


def test_masked_tokens_and_equal_rows():
    rng = np.random.default_rng(3)
    V = 20000
    x = rng.normal(0, 2, size=(3, V)).astype(np.float32)
    x[0, rng.random(V) < 0.9] = -np.inf     # most tokens masked
    x[1, :] = 0.5                           # every logit equal: ids 0..k-1, p = 1/V
    x[2, :] = -np.inf
    x[2, 12345] = 3.0                       # one live token: p = 1 there, 0 elsewhere
    seen, ids, probs, z, lse = _run(x, 256)
    _check(seen, 256, ids, probs, z, lse)
    assert ids[1].tolist() == list(range(256))
    assert ids[2, 0] == 12345 and abs(probs[2, 0] - 1.0) < 1e-6


def test_unlucky_sample_takes_the_slices():
    # every raised logit sits in a sampled chunk (chunks 0, 16, 32, ... of 128
    # tokens), so the sampled bound is high and fewer than k tokens reach it:
    # the row must take the exact slice path
    rng = np.random.default_rng(5)
    V = 128256
    x = rng.normal(0, 1, size=(2, V)).astype(np.float32)
    sampled = np.array([c * 2048 + o for c in range(V // 2048) for o in range(128)])
    for r in range(2):
        hot = rng.choice(sampled, size=200, replace=False)
        x[r, hot] = 10.0 + rng.random(200).astype(np.float32)
    seen, ids, probs, z, lse = _run(x, 256)
    _check(seen, 256, ids, probs, z, lse)


def test_crowded_tie_at_the_kth_value():
    # 3,000 copies of the k-th largest value: the merge's window bin of that
    # value overflows its places and the exact select breaks the tie by token
    rng = np.random.default_rng(6)
    V = 128256
    x = rng.normal(0, 1, size=(2, V)).astype(np.float32)
    for r in range(2):
        x[r, rng.choice(V, size=3000, replace=False)] = 5.0
        x[r, rng.choice(V, size=100, replace=False)] = 8.0
    seen, ids, probs, z, lse = _run(x, 256)
    _check(seen, 256, ids, probs, z, lse)


def test_back_to_back_calls_share_a_workspace():
    # calls queued one after another on one stream with one workspace and no
    # host synchronization between them: each call's kernels start while the
    # previous call's drain, and every result must still be its own
    import torch
    from programmable_paged_kv_gb300 import readout_topk, readout_topk_workspace_bytes
    from programmable_paged_kv_gb300.abi import PIE_F32
    R, V, k = 4, 40000, 256
    rng = np.random.default_rng(8)
    arrays = [W.readout_logits(20 + i, R, V, spikes=4) for i in range(3)]
    x = rng.normal(0, 2, size=(R, V)).astype(np.float32)
    x[1, :] = 0.25                          # a row for the slices
    x[2, rng.random(V) < 0.95] = -np.inf    # mostly masked
    arrays.insert(1, x)
    ws = torch.empty(readout_topk_workspace_bytes(PIE_F32, R, V, k), dtype=torch.uint8,
                     device="cuda")
    devs = [torch.from_numpy(a).cuda() for a in arrays]
    outs = [(torch.empty((R, k), dtype=torch.int32, device="cuda"),
             torch.empty((R, k), dtype=torch.float32, device="cuda"),
             torch.empty(R, dtype=torch.float32, device="cuda"),
             torch.empty(R, dtype=torch.float32, device="cuda")) for _ in arrays]
    torch.cuda.synchronize()
    for dev, o in zip(devs, outs):  # kernels only between the calls
        readout_topk(dev, k, *o, workspace=ws)
    torch.cuda.synchronize()
    for a, o in zip(arrays, outs):
        _check(a, k, *(t.cpu().numpy() for t in o))
