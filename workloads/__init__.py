"""Seeded synthetic inputs for one Pie ForwardPass attention layer.

This module only *describes* workloads: the lanes, their rows and page
tables, the StateGeometry fields (positions, slots, kv_len, fold), the
per-row slot masks, and the q/k/v and cached K/V values drawn from a seeded
N(0, 1).  It holds none of the method's arithmetic (no RoPE, no attention,
no fold), so that both the CPU oracle and the CUDA library can be fed from
it without sharing any computation.

The shapes follow the use cases on the Pie "The forward pass" page (Lanes:
guidance lane pairs; State geometry: folding() and speculative drafts with a
device-channel fold; Attention masks: sliding window, sinks, TOVA eviction;
Readouts: last row per lane or a whole draft window) and the KvPage size of
8-32 tokens from the Pie review (section 2.1).

Storage conventions shared by every consumer:
  * float32 tensors are numpy float32 arrays;
  * bfloat16 tensors are numpy uint16 arrays holding the bf16 bit patterns;
  * K/V pools are laid out [num_pages][num_kv_heads][page_size][head_dim];
  * a row's mask words are LSB-first: slot s of row r is visible iff bit
    (s & 31) of mask_words[mask_word_indptr[r] + (s >> 5)] is set.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np

F32 = 0
BF16 = 1
DTYPE_NAMES = {F32: "f32", BF16: "bf16"}
ELEM_BYTES = {F32: 4, BF16: 2}

FOLD_NONE = 0
FOLD_ALL = 1
FOLD_COUNT = 2
FOLD_CHANNEL = 3

# Bit patterns written into never-written pool slots.  Both are NaN, so a
# kernel that reads a slot it must not read poisons its output visibly.
CANARY = {F32: np.uint32(0xFFFFFFFF), BF16: np.uint16(0xFFFF)}


# --------------------------------------------------------------------------
# dtype helpers (data preparation only)
# --------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest even); return bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = np.uint16(0x7FC0)
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def to_storage(x: np.ndarray, dtype: int) -> np.ndarray:
    if dtype == F32:
        return np.ascontiguousarray(x, dtype=np.float32)
    return f32_to_bf16_bits(x)


def storage_to_f32(x: np.ndarray, dtype: int) -> np.ndarray:
    if dtype == F32:
        return np.ascontiguousarray(x, dtype=np.float32)
    return bf16_bits_to_f32(x)


def storage_np_dtype(dtype: int):
    return np.float32 if dtype == F32 else np.uint16


def canary_array(shape, dtype: int) -> np.ndarray:
    """A storage array whose every element is the dtype's canary bit pattern."""
    if dtype == F32:
        return np.full(shape, CANARY[F32], dtype=np.uint32).view(np.float32)
    return np.full(shape, CANARY[BF16], dtype=np.uint16)


# --------------------------------------------------------------------------
# Workload description
# --------------------------------------------------------------------------
@dataclasses.dataclass
class Desc:
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    dtype: int
    rope_base: float = 10000.0
    sm_scale: float = 0.0  # 0 means 1/sqrt(head_dim)


@dataclasses.dataclass
class Pass:
    """One ForwardPass: the lanes' rows, their StateGeometry and inputs."""
    row_indptr: np.ndarray          # int32 [L+1]
    positions: np.ndarray           # int32 [N]
    slots: np.ndarray               # int32 [N]
    kv_len: np.ndarray              # int32 [L]
    page_indptr: np.ndarray         # int32 [L+1]
    page_ids: np.ndarray            # int32 [page_indptr[L]] physical page ids
    fold_mode: np.ndarray           # int32 [L]
    fold_count: np.ndarray          # int32 [L] (used by FOLD_COUNT)
    q: np.ndarray                   # storage [N, Hq, d]
    k: np.ndarray                   # storage [N, Hkv, d]
    v: np.ndarray                   # storage [N, Hkv, d]
    mask_word_indptr: Optional[np.ndarray] = None  # int64 [N+1]
    mask_words: Optional[np.ndarray] = None        # uint32
    readout: Optional[np.ndarray] = None           # int32 [R]
    channel: Optional[np.ndarray] = None           # int32 [L], value the epilogue writes

    @property
    def num_lanes(self) -> int:
        return int(self.kv_len.shape[0])

    @property
    def num_rows(self) -> int:
        return int(self.positions.shape[0])


@dataclasses.dataclass
class Scenario:
    """A pool, its initial contents, and a sequence of passes on one stream."""
    name: str
    desc: Desc
    num_pool_pages: int
    pool_pages: np.ndarray          # int32 sorted distinct physical pages referenced
    k_init: np.ndarray              # storage [U, Hkv, P, d] for pool_pages
    v_init: np.ndarray              # storage [U, Hkv, P, d]
    frozen_len0: np.ndarray         # int32 [L]
    passes: List[Pass]
    recipe: str = ""

    def compact_page_ids(self, page_ids: np.ndarray) -> np.ndarray:
        """Map physical page ids to indices into pool_pages (k_init/v_init)."""
        idx = np.searchsorted(self.pool_pages, page_ids)
        assert np.all(self.pool_pages[idx] == page_ids)
        return idx.astype(np.int32)


# --------------------------------------------------------------------------
# generators
# --------------------------------------------------------------------------
def _rngs(seed: int, n: int):
    return [np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(n)]


def _normal(rng, shape, dtype):
    return to_storage(rng.standard_normal(size=shape, dtype=np.float32), dtype)


def _pack_mask(visible: np.ndarray) -> np.ndarray:
    """bool [rows, kv] -> uint32 [rows, ceil(kv/32)] LSB-first words."""
    rows, kv = visible.shape
    nw = (kv + 31) // 32
    padded = np.zeros((rows, nw * 32), dtype=bool)
    padded[:, :kv] = visible
    b = np.packbits(padded, axis=1, bitorder="little")  # [rows, nw*4] bytes
    w = b.view("<u4").astype(np.uint32)
    return np.ascontiguousarray(w.reshape(rows, nw))


def mask_from_visible(visible_rows: List[np.ndarray]):
    """Per-row bool arrays (length kv_len of the row's lane) -> indptr, words."""
    words = []
    indptr = [0]
    for vis in visible_rows:
        w = _pack_mask(vis.reshape(1, -1))[0] if vis.size else np.zeros(0, np.uint32)
        words.append(w)
        indptr.append(indptr[-1] + w.size)
    allw = np.concatenate(words) if words else np.zeros(0, np.uint32)
    return np.asarray(indptr, np.int64), allw.astype(np.uint32)


# When False, generators leave a scenario's cached K/V unset (k_init and
# v_init are None): the metadata and the per-row q/k/v are drawn as usual,
# and whoever runs the scenario fills the pool pages itself (the benchmark
# does so on the device with the same N(0,1) distribution, which is much
# faster than drawing hundreds of MB on the host).  See geometry_only().
_POOL_DATA = True


class geometry_only:
    """Context in which generators skip drawing the cached pool contents."""

    def __enter__(self):
        global _POOL_DATA
        self._old, _POOL_DATA = _POOL_DATA, False
        return self

    def __exit__(self, *exc):
        global _POOL_DATA
        _POOL_DATA = self._old
        return False


def _fill_pool_init(desc: Desc, pool_pages: np.ndarray, lane_pages, cached, rng):
    """Random cached K/V for slots [0, cached[l]) of each lane; canary elsewhere.

    lane_pages[l] are the lane's physical pages in slot order.  Pages shared by
    several lanes are filled once (by the first lane that lists them).  Inside
    geometry_only() nothing is drawn and (None, None) is returned.
    """
    if not _POOL_DATA:
        return None, None
    U = pool_pages.size
    H, P, d = desc.num_kv_heads, desc.page_size, desc.head_dim
    k = canary_array((U, H, P, d), desc.dtype)
    v = canary_array((U, H, P, d), desc.dtype)
    done = set()
    for l, pages in enumerate(lane_pages):
        c = int(cached[l])
        for j, pg in enumerate(pages):
            pg = int(pg)
            if pg in done:
                continue
            nslot = min(P, max(0, c - j * P))
            if nslot == 0:
                continue
            done.add(pg)
            u = int(np.searchsorted(pool_pages, pg))
            k[u, :, :nslot, :] = _normal(rng, (H, nslot, d), desc.dtype)
            v[u, :, :nslot, :] = _normal(rng, (H, nslot, d), desc.dtype)
    return k, v


def _lane_pass(desc, lane_rows, lane_pages, kv_len, fold_mode, rng, fold_count=None,
               mask_rows=None, readout=None, channel=None):
    """Assemble a Pass from per-lane (positions, slots) lists."""
    L = len(lane_rows)
    row_indptr = np.zeros(L + 1, np.int32)
    for l, (pos, _) in enumerate(lane_rows):
        row_indptr[l + 1] = row_indptr[l] + len(pos)
    N = int(row_indptr[-1])
    positions = np.concatenate([np.asarray(p, np.int32) for p, _ in lane_rows]) if N else np.zeros(0, np.int32)
    slots = np.concatenate([np.asarray(s, np.int32) for _, s in lane_rows]) if N else np.zeros(0, np.int32)
    page_indptr = np.zeros(L + 1, np.int32)
    for l, pages in enumerate(lane_pages):
        page_indptr[l + 1] = page_indptr[l] + len(pages)
    page_ids = (np.concatenate([np.asarray(p, np.int32) for p in lane_pages])
                if page_indptr[-1] else np.zeros(0, np.int32))
    Hq, Hkv, d = desc.num_q_heads, desc.num_kv_heads, desc.head_dim
    q = _normal(rng, (N, Hq, d), desc.dtype)
    k = _normal(rng, (N, Hkv, d), desc.dtype)
    v = _normal(rng, (N, Hkv, d), desc.dtype)
    fm = np.asarray(fold_mode, np.int32)
    fc = np.zeros(L, np.int32) if fold_count is None else np.asarray(fold_count, np.int32)
    mwi = mw = None
    if mask_rows is not None:
        mwi, mw = mask_from_visible(mask_rows)
    return Pass(row_indptr=row_indptr, positions=positions, slots=slots,
                kv_len=np.asarray(kv_len, np.int32), page_indptr=page_indptr,
                page_ids=page_ids, fold_mode=fm, fold_count=fc, q=q, k=k, v=v,
                mask_word_indptr=mwi, mask_words=mw,
                readout=None if readout is None else np.asarray(readout, np.int32),
                channel=None if channel is None else np.asarray(channel, np.int32))


def _permuted_pool(rng, num_pool_pages, counts):
    """Disjoint consecutive chunks of one random permutation of page ids."""
    perm = rng.permutation(num_pool_pages).astype(np.int32)
    out, o = [], 0
    for c in counts:
        out.append(perm[o:o + c])
        o += c
    assert o <= num_pool_pages
    return out


def _pages_for(n_slots, P):
    return (n_slots + P - 1) // P


# ---- configuration 1: tiny fp32 single-layer forward --------------------------
def tiny(seed: int = 0, prompt: int = 40, decodes: int = 8) -> Scenario:
    """1 lane, 4 q / 2 kv heads, d=64, fp32, P=16: a folding() prefill of the
    prompt followed by single-row decode passes (Pie review Algorithm 1)."""
    desc = Desc(4, 2, 64, 16, F32)
    r_meta, r_data = _rngs(seed, 2)
    T = prompt + decodes
    npages = _pages_for(T, desc.page_size)
    pool = 8 if npages <= 8 else npages
    (pages,) = _permuted_pool(r_meta, pool, [npages])
    # all 48 tokens' q/k/v drawn up front so that prefix+continuation and a
    # monolithic pass see the same inputs
    Q = _normal(r_data, (T, 4, 64), F32)
    K = _normal(r_data, (T, 2, 64), F32)
    V = _normal(r_data, (T, 2, 64), F32)
    passes = []
    spans = [(0, prompt)] + [(prompt + i, prompt + i + 1) for i in range(decodes)]
    for a, b in spans:
        p = _lane_pass(desc, [(np.arange(a, b), np.arange(a, b))], [pages], [b],
                       [FOLD_ALL], r_meta)
        p.q, p.k, p.v = Q[a:b].copy(), K[a:b].copy(), V[a:b].copy()
        passes.append(p)
    pool_pages = np.sort(pages)
    k0, v0 = _fill_pool_init(desc, pool_pages, [pages], [0], r_data)
    return Scenario("tiny", desc, pool, pool_pages, k0, v0, np.zeros(1, np.int32), passes,
                    recipe="q/k/v ~ N(0,1) fp32 for all 48 tokens; 40-row folding() "
                           "prefill then 8 single-row decodes; 3 of 8 pages, permuted")


# ---- configuration 2: decode batch ---------------------------------------------
def decode_batch(seed: int = 0, lanes: int = 64, c_lo: int = 512, c_hi: int = 4096,
                 num_pool_pages: int = 65536, desc: Optional[Desc] = None) -> Scenario:
    """64 lanes x 1 row; cached length C ~ U[512, 4096]; row at position/slot C;
    kv_len C+1; fold=all; pages randomly permuted in a 64k-page pool."""
    desc = desc or Desc(32, 8, 128, 16, BF16)
    r_meta, r_data = _rngs(seed, 2)
    C = r_meta.integers(c_lo, c_hi + 1, size=lanes).astype(np.int32)
    counts = [_pages_for(int(c) + 1, desc.page_size) for c in C]
    lane_pages = _permuted_pool(r_meta, num_pool_pages, counts)
    p = _lane_pass(desc, [([c], [c]) for c in C], lane_pages, C + 1,
                   [FOLD_ALL] * lanes, r_data)
    pool_pages = np.sort(np.concatenate(lane_pages))
    k0, v0 = _fill_pool_init(desc, pool_pages, lane_pages, C, r_data)
    return Scenario("decode_batch", desc, num_pool_pages, pool_pages, k0, v0, C.copy(), [p],
                    recipe=f"{lanes} lanes x 1 row, C ~ U[{c_lo},{c_hi}], cached K/V and "
                           "q/k/v ~ N(0,1) bf16, pages permuted")


def decode_loop_meta(seed: int = 0, lanes: int = 64, steps: int = 64, c_lo: int = 512,
                     c_hi: int = 4096, num_pool_pages: int = 65536,
                     desc: Optional[Desc] = None):
    """The decode batch continued for `steps` single-row passes: pass t puts
    each lane's row at position/slot C+t, reads C+t+1 slots and folds it.
    Returns (desc, C, lane_pages, pass_meta(t) -> Pass without q/k/v)."""
    desc = desc or Desc(32, 8, 128, 16, BF16)
    r_meta = _rngs(seed, 2)[0]
    C = r_meta.integers(c_lo, c_hi + 1, size=lanes).astype(np.int32)
    counts = [_pages_for(int(c) + steps, desc.page_size) for c in C]
    lane_pages = _permuted_pool(r_meta, num_pool_pages, counts)
    page_indptr = np.zeros(lanes + 1, np.int32)
    page_indptr[1:] = np.cumsum(counts)
    page_ids = np.concatenate(lane_pages).astype(np.int32)
    e = np.zeros((0,), np.uint16)

    def pass_meta(t: int) -> Pass:
        pos = (C + t).astype(np.int32)
        return Pass(row_indptr=np.arange(lanes + 1, dtype=np.int32), positions=pos,
                    slots=pos.copy(), kv_len=(pos + 1).astype(np.int32),
                    page_indptr=page_indptr, page_ids=page_ids,
                    fold_mode=np.full(lanes, FOLD_ALL, np.int32),
                    fold_count=np.zeros(lanes, np.int32), q=e, k=e, v=e)

    return desc, C, lane_pages, pass_meta


def decode_loop(seed: int = 0, lanes: int = 64, steps: int = 8, c_lo: int = 512,
                c_hi: int = 4096, num_pool_pages: int = 65536, desc: Optional[Desc] = None,
                spare: int = 0) -> Scenario:
    """The decode batch as `steps` single-row passes with q/k/v: pass t puts
    each lane's row at position/slot C+t, reads C+t+1 slots and folds it.
    Each lane's pages hold C + steps + spare slots (rounded up to pages)."""
    desc = desc or Desc(32, 8, 128, 16, BF16)
    r_meta, r_data = _rngs(seed, 2)
    C = r_meta.integers(c_lo, c_hi + 1, size=lanes).astype(np.int32)
    counts = [_pages_for(int(c) + steps + spare, desc.page_size) for c in C]
    lane_pages = _permuted_pool(r_meta, num_pool_pages, counts)
    passes = [_lane_pass(desc, [([int(c) + t], [int(c) + t]) for c in C], lane_pages, C + t + 1,
                         [FOLD_ALL] * lanes, r_data) for t in range(steps)]
    pool_pages = np.sort(np.concatenate(lane_pages))
    k0, v0 = _fill_pool_init(desc, pool_pages, lane_pages, C, r_data)
    return Scenario("decode_loop", desc, num_pool_pages, pool_pages, k0, v0, C.copy(), passes,
                    recipe=f"{lanes} lanes x {steps} single-row steps, C ~ U[{c_lo},{c_hi}]")


# ---- configuration 3: guidance lane pairs ---------------------------------------
def guidance_pairs(seed: int = 0, pairs: int = 32, prefix: int = 1024, prefill: int = 64,
                   decodes: int = 16, num_pool_pages: int = 4096,
                   desc: Optional[Desc] = None) -> Scenario:
    """cond/uncond lane pairs sharing a frozen prefix of pages; each lane
    prefills `prefill` causal rows then decodes; readout = last row per lane."""
    desc = desc or Desc(32, 8, 128, 32, BF16)
    P = desc.page_size
    assert prefix % P == 0
    r_meta, r_data = _rngs(seed, 2)
    total = prefix + prefill + decodes
    shared_n = prefix // P
    priv_n = _pages_for(total, P) - shared_n
    chunks = _permuted_pool(r_meta, num_pool_pages, [shared_n + 2 * priv_n] * pairs)
    lane_pages = []
    for ch in chunks:
        shared = ch[:shared_n]
        lane_pages.append(np.concatenate([shared, ch[shared_n:shared_n + priv_n]]))
        lane_pages.append(np.concatenate([shared, ch[shared_n + priv_n:]]))
    L = 2 * pairs
    passes = []
    spans = [(prefix, prefix + prefill)] + [(prefix + prefill + t, prefix + prefill + t + 1)
                                           for t in range(decodes)]
    for a, b in spans:
        rows = [(np.arange(a, b), np.arange(a, b)) for _ in range(L)]
        passes.append(_lane_pass(desc, rows, lane_pages, [b] * L, [FOLD_ALL] * L, r_data))
    pool_pages = np.sort(np.unique(np.concatenate(lane_pages)))
    k0, v0 = _fill_pool_init(desc, pool_pages, lane_pages, [prefix] * L, r_data)
    return Scenario("guidance_pairs", desc, num_pool_pages, pool_pages, k0, v0,
                    np.full(L, prefix, np.int32), passes,
                    recipe=f"{pairs} lane pairs sharing a {prefix}-token prefix ({shared_n} "
                           f"pages of {P}); {prefill} causal prefill rows per lane then "
                           f"{decodes} decodes; q/k/v ~ N(0,1) bf16")


# ---- configuration 4: speculative verify ----------------------------------------
def spec_verify(seed: int = 0, lanes: int = 48, draft: int = 8, c_lo: int = 1024,
                c_hi: int = 8192, num_pool_pages: int = 32768,
                desc: Optional[Desc] = None) -> Scenario:
    """Each lane writes `draft` unfrozen rows at C..C+draft-1, reads out all of
    them, then folds the accepted count a ~ U{0..draft} from a device channel;
    a follow-up decode at slot C+a overwrites the first rejected draft."""
    desc = desc or Desc(32, 8, 128, 16, BF16)
    r_meta, r_data = _rngs(seed, 2)
    C = r_meta.integers(c_lo, c_hi + 1, size=lanes).astype(np.int32)
    a = r_meta.integers(0, draft + 1, size=lanes).astype(np.int32)
    counts = [_pages_for(int(c) + draft, desc.page_size) for c in C]
    lane_pages = _permuted_pool(r_meta, num_pool_pages, counts)
    rows = [(np.arange(c, c + draft), np.arange(c, c + draft)) for c in C]
    N = lanes * draft
    p1 = _lane_pass(desc, rows, lane_pages, C + draft, [FOLD_CHANNEL] * lanes, r_data,
                    readout=np.arange(N, dtype=np.int32), channel=a)
    F = C + a
    p2 = _lane_pass(desc, [([f], [f]) for f in F], lane_pages, F + 1, [FOLD_ALL] * lanes, r_data)
    pool_pages = np.sort(np.concatenate(lane_pages))
    k0, v0 = _fill_pool_init(desc, pool_pages, lane_pages, C, r_data)
    return Scenario("spec_verify", desc, num_pool_pages, pool_pages, k0, v0, C.copy(), [p1, p2],
                    recipe=f"{lanes} lanes, C ~ U[{c_lo},{c_hi}], {draft} draft rows with "
                           f"fold from a channel a ~ U{{0..{draft}}}, readout of all drafts, "
                           "then one decode at C+a")


# ---- configuration 5: masked long context ----------------------------------------
def masked_long(seed: int = 0, kind: str = "window", lanes: int = 8, kv: int = 32768,
                rows: int = 64, sinks: int = 4, window: int = 4096, keep: float = 0.25,
                desc: Optional[Desc] = None) -> Scenario:
    """`rows` prefill rows at the end of a `kv`-slot working set; per-row masks:
    'window' = first `sinks` slots + the last `window` slots up to the row's own
    slot; 'tova' = a Bernoulli(keep) subset of the cached slots, shared by all
    rows of the lane, plus causal visibility of the new rows."""
    desc = desc or Desc(32, 8, 128, 16, BF16)
    r_meta, r_data = _rngs(seed, 2)
    C = kv - rows
    npages = _pages_for(kv, desc.page_size)
    lane_pages = _permuted_pool(r_meta, lanes * npages, [npages] * lanes)
    vis_rows = []
    s = np.arange(kv)
    for l in range(lanes):
        if kind == "tova":
            kept = r_meta.random(C) < keep
        for i in range(rows):
            p = C + i
            if kind == "window":
                vis = (s < sinks) | ((s <= p) & (s > p - window))
            elif kind == "tova":
                vis = np.zeros(kv, bool)
                vis[:C] = kept
                vis[C:p + 1] = True
            else:
                raise ValueError(kind)
            vis_rows.append(vis)
    lr = [(np.arange(C, kv), np.arange(C, kv)) for _ in range(lanes)]
    p1 = _lane_pass(desc, lr, lane_pages, [kv] * lanes, [FOLD_ALL] * lanes, r_data,
                    mask_rows=vis_rows)
    pool_pages = np.sort(np.concatenate(lane_pages))
    k0, v0 = _fill_pool_init(desc, pool_pages, lane_pages, [C] * lanes, r_data)
    rec = (f"{lanes} lanes, {rows} rows at slots {C}..{kv-1}, " +
           (f"{sinks} sinks + {window}-slot window" if kind == "window"
            else f"TOVA keep {keep} Bernoulli per cached slot") + ", q/k/v ~ N(0,1) bf16")
    return Scenario(f"masked_{kind}", desc, lanes * npages, pool_pages, k0, v0,
                    np.full(lanes, C, np.int32), [p1], recipe=rec)


# ---- small variants spanning several tiles and a ragged tail -----------------------
def small(name: str, seed: int = 0) -> Scenario:
    """Reduced copies of the five configurations that the oracle finishes in
    seconds while still covering several KV tiles, ragged lanes and tails."""
    if name == "tiny":
        return tiny(seed)
    if name == "decode_batch":
        return decode_batch(seed, lanes=9, c_lo=1, c_hi=700, num_pool_pages=1024)
    if name == "guidance_pairs":
        return guidance_pairs(seed, pairs=3, prefix=96, prefill=40, decodes=3,
                              num_pool_pages=256)
    if name == "spec_verify":
        return spec_verify(seed, lanes=5, c_lo=17, c_hi=600, num_pool_pages=512)
    if name == "masked_window":
        return masked_long(seed, "window", lanes=2, kv=1100, rows=40, window=300)
    if name == "masked_tova":
        return masked_long(seed, "tova", lanes=2, kv=1100, rows=40)
    if name == "masked_decode_window":
        return masked_long(seed, "window", lanes=3, kv=1300, rows=1, window=300)
    if name == "masked_decode_tova":
        return masked_long(seed, "tova", lanes=3, kv=1300, rows=1)
    raise ValueError(name)


def readout_logits(seed: int, rows: int, vocab: int, spikes: int = 8,
                   scale: float = 2.0) -> np.ndarray:
    """Synthetic next-token logits for the readout epilogue, float32 [rows,
    vocab]: N(0, scale) per token plus `spikes` tokens per row raised by
    U[6, 14] (a peaked distribution, like a language model's; no trained
    weights)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 7]))
    x = rng.normal(0.0, scale, size=(rows, vocab)).astype(np.float32)
    for r in range(rows):
        idx = rng.choice(vocab, size=min(spikes, vocab), replace=False)
        x[r, idx] += rng.uniform(6.0, 14.0, size=idx.size).astype(np.float32)
    return x


@dataclasses.dataclass
class AdapterSite:
    """Inputs of the adapters at one projection site: the lanes' rows and
    adapter ids, x [N, d_in] and y [N, d_out] (bf16 bit patterns), the
    adapters' A [n_ad, r, d_in], B [n_ad, d_out, r] (bf16 bits), scale
    float32 [n_ad] and IA3 vectors [n_ad, d_out] (bf16 bits) or None."""
    row_indptr: np.ndarray
    adapter_of_lane: np.ndarray
    x: np.ndarray
    y: np.ndarray
    lora_a: Optional[np.ndarray]
    lora_b: Optional[np.ndarray]
    scale: np.ndarray
    ia3: Optional[np.ndarray]
    rank: int
    recipe: str


def adapter_site(seed: int, rows_per_lane, n_adapters: int = 16, d_in: int = 4096,
                 d_out: int = 4096, rank: int = 16, ia3: bool = True,
                 none_every: int = 8) -> AdapterSite:
    """Synthetic per-lane adapters (no trained weights): every lane draws an
    adapter uniformly from n_adapters, except every `none_every`-th lane,
    which has none (-1); x, y ~ N(0, 1); A ~ N(0, 1/d_in) and B ~ N(0, 1/r)
    so that B (A x) is of the order of y; scale = 2 (LoRA alpha = 2 r);
    IA3 entries ~ U[0.5, 1.5].  rank 0 gives an IA3-only site."""
    rows = np.asarray(rows_per_lane, dtype=np.int64).reshape(-1)
    L = rows.size
    rng = np.random.default_rng(np.random.SeedSequence([seed, 11]))
    row_indptr = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    N = int(row_indptr[-1])
    ad = rng.integers(0, max(n_adapters, 1), size=L).astype(np.int32)
    if none_every > 0:
        ad[none_every - 1::none_every] = -1
    if n_adapters == 0:
        ad[:] = -1
    f32 = np.float32
    x = f32_to_bf16_bits(rng.standard_normal((N, d_in), dtype=f32))
    y = f32_to_bf16_bits(rng.standard_normal((N, d_out), dtype=f32))
    a = b = None
    if rank > 0:
        a = f32_to_bf16_bits(rng.standard_normal((n_adapters, rank, d_in), dtype=f32) / f32(np.sqrt(d_in)))
        b = f32_to_bf16_bits(rng.standard_normal((n_adapters, d_out, rank), dtype=f32) / f32(np.sqrt(rank)))
    scale = np.full(n_adapters, 2.0, dtype=f32)
    s = f32_to_bf16_bits(rng.uniform(0.5, 1.5, size=(n_adapters, d_out)).astype(f32)) if ia3 else None
    recipe = (f"{L} lanes, {N} rows, adapter per lane ~ U{{0..{n_adapters - 1}}} (every "
              f"{none_every}th lane none), d_in {d_in}, d_out {d_out}, rank {rank}, "
              f"x, y ~ N(0,1), A ~ N(0,1/d_in), B ~ N(0,1/r), scale 2, "
              f"IA3 {'~ U[0.5,1.5]' if ia3 else 'off'}, bf16")
    return AdapterSite(row_indptr, ad, x, y, a, b, scale, s, rank, recipe)


@dataclasses.dataclass
class CallTrace:
    """GPU-bound forward calls from several command queues, in arrival order,
    for the work-conserving batcher: queue q owns one working set (its pages
    in slot order, frozen for its first cached[q] slots); each call appends n
    rows to its queue's working set (the folding() geometry: position = slot
    = the next free slot, fold all).  `pool` holds the pages' initial
    contents (passes is empty)."""
    pool: Scenario
    queue_pages: List[np.ndarray]
    cached: np.ndarray               # int32 [Q]
    priority: np.ndarray             # int32 [Q]
    calls: list                      # [(queue, q [n,Hq,d], k [n,Hkv,d], v [n,Hkv,d])]
    recipe: str = ""


def forward_calls(seed: int = 0, queues: int = 16, calls_per_queue: int = 6, prefix: int = 256,
                  private_hi: int = 100, prefill_lo: int = 8, prefill_hi: int = 64,
                  desc: Optional[Desc] = None, num_pool_pages: int = 4096) -> CallTrace:
    """Queues 2i and 2i+1 share a frozen prefix of `prefix` slots (whole
    pages, read-only) and add U[0, private_hi] cached slots of their own; each
    queue's first call is a prefill of U[prefill_lo, prefill_hi] rows, the
    others decode steps (one row) or short continuations (U[2, 8] rows); the
    calls of all queues arrive interleaved in a seeded random order, queue
    priorities ~ U{0, 1, 2}; q/k/v ~ N(0, 1)."""
    desc = desc or Desc(32, 8, 128, 16, BF16)
    P = desc.page_size
    assert prefix % P == 0
    rng = np.random.default_rng(np.random.SeedSequence([seed, 13]))
    extra = rng.integers(0, private_hi + 1, size=queues)
    rows = []
    for q in range(queues):
        r = [int(rng.integers(prefill_lo, prefill_hi + 1))]
        for _ in range(calls_per_queue - 1):
            r.append(1 if rng.random() < 0.6 else int(rng.integers(2, 9)))
        rows.append(r)
    npairs = (queues + 1) // 2
    shared_pages = prefix // P
    private_need = [_pages_for(int(extra[q]) + sum(rows[q]), P) + 1 for q in range(queues)]
    chunks = _permuted_pool(rng, num_pool_pages, [shared_pages] * npairs + private_need)
    queue_pages = []
    for q in range(queues):
        queue_pages.append(np.concatenate([chunks[q // 2], chunks[npairs + q]]).astype(np.int32))
    cached = (prefix + extra).astype(np.int32)
    pool_pages = np.unique(np.concatenate(queue_pages)).astype(np.int32)
    k_init, v_init = _fill_pool_init(desc, pool_pages, queue_pages, cached, rng)
    order = np.concatenate([np.full(calls_per_queue, q) for q in range(queues)])
    rng.shuffle(order)
    seen = np.zeros(queues, np.int64)
    calls = []
    Hq, Hkv, d = desc.num_q_heads, desc.num_kv_heads, desc.head_dim
    for q in order:
        n = rows[q][seen[q]]
        seen[q] += 1
        calls.append((int(q), _normal(rng, (n, Hq, d), desc.dtype),
                      _normal(rng, (n, Hkv, d), desc.dtype), _normal(rng, (n, Hkv, d), desc.dtype)))
    pool = Scenario("forward_calls", desc, num_pool_pages, pool_pages, k_init, v_init, cached, [],
                    "")
    recipe = (f"{queues} queues x {calls_per_queue} calls, pairs share a {prefix}-slot prefix, "
              f"private cached U[0,{private_hi}], prefill U[{prefill_lo},{prefill_hi}] rows then "
              f"decodes (60%) or 2-8-row continuations, random interleaving, priorities U{{0,1,2}}")
    return CallTrace(pool, queue_pages, cached, rng.integers(0, 3, size=queues).astype(np.int32),
                     calls, recipe)


FULL = {
    "tiny": lambda seed=0: tiny(seed),
    "decode_batch": lambda seed=0: decode_batch(seed),
    "guidance_pairs": lambda seed=0: guidance_pairs(seed),
    "spec_verify": lambda seed=0: spec_verify(seed),
    "masked_window": lambda seed=0: masked_long(seed, "window"),
    "masked_tova": lambda seed=0: masked_long(seed, "tova"),
    # masked decode: one row per lane at the end of the same working sets
    "masked_decode_window": lambda seed=0: masked_long(seed, "window", rows=1),
    "masked_decode_tova": lambda seed=0: masked_long(seed, "tova", rows=1),
}
SMALL_NAMES = list(FULL.keys())
