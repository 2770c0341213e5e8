// Step 2-3 of a ForwardPass for lanes with many query vectors per kv head
// (prefill rows, speculative-verify drafts, masked prefill): grouped-query
// attention over paged K/V on the 5th-generation tensor cores (Pie "The
// forward pass": State geometry kv_len; Attention masks; Readouts).
//
// One CTA handles a work item: NT (1 or 2) tiles of 128 query vectors (the G
// heads of a kv group for 128/G consecutive rows of one lane per tile,
// head-minor) against one chunk of the lane's slots, in KV tiles of BN slots
// (128 with one query tile, 64 with two, so that two score buffers per query
// tile and every tile's O fit the 512 TMEM columns).  With NT = 2 both query
// tiles share every K/V tile, so the chunk is read once for 256 query vectors.
//   warps 0, 1  TMA producers, K and V: the query tiles once (4-D tensor map
//            over q_rot viewed as [N][Hkv][G][d]), then per KV tile the K (V)
//            block of every page in the tile (2-D tensor maps over the pools,
//            one 64-column box per half of d, 128-byte swizzle) into an
//            NS-deep ring of stages, each copy from its own lane (a warp's
//            copies issue one after another); in masked passes, whole pages
//            of a page-granular slot list the same way, and the rows of a
//            slot-granular list with tile::gather4.  K and V land on
//            separate barriers, so scores wait for K only;
//   warps 2..1+NT  one MMA issuer per query tile t (warp 2 also allocates the
//            512 TMEM columns): from one thread, S_t = Q_t K^T (M=128, N=BN)
//            into one of two score buffers and O_t += P_t V (M=128, N=128,
//            K=BN) with P_t read from TMEM, where the softmax stored it over
//            the first half of the score buffer.  Scores for KV tile j+2 are
//            issued right after P.V of tile j (the in-order tensor pipe
//            guarantees that P is read first), so the softmax of tile j+1
//            never waits for them; two issuers keep both tiles' chains in
//            flight at once;
//   warps 2+NT.. one 4-warp softmax group per query tile: each thread owns one
//            query row (its TMEM lane), loads its BN scores with one
//            tcgen05.ld, applies the row's visibility (slot-causal or its
//            mask words; tiles visible in full skip the per-column test),
//            keeps the online max/sum in the log2 domain (the max used for
//            the exponent only moves when the tile max exceeds it by more
//            than 2^8, so O is rarely rescaled), rescales O in TMEM when it
//            does move, and stores P as bf16 pairs into TMEM.  Warps whose
//            32 query rows are all padding skip the work.
// At the end each thread writes its row's output: normalised to bf16 plus lse
// when the item covers the row's whole visible range, else its partial state
// (max, sum, unnormalised output) for the combine step.  Every wait is
// bounded in time.

#include "common.cuh"
#include "tc_util.cuh"
#include "tmem128.cuh"

namespace pie {

namespace tc {

constexpr int kQHalf = 128 * 128;        // 128 query rows x 128 bytes (half of d)

// Tile geometry per number of query tiles.  TMEM holds two score buffers per
// query tile plus each tile's 128-column O: one query tile takes 128-slot KV
// tiles (2 x 128 + 128 columns), two query tiles 64-slot ones (4 x 64 + 256).
template <int NT>
struct Cfg {
  static constexpr int BN = tc_kv_tile(NT);         // KV slots per tile
  static constexpr int kKvHalf = BN * 128;          // BN slot rows x 128 bytes (half of d)
  static constexpr int NS = NT == 1 ? 3 : 4;        // KV stages beside the query tiles
  static constexpr int kIssuer0 = 2;                // warps 0, 1: K and V producers
  static constexpr int kIssuers = NT;               // one MMA-issuing warp per query tile
  static constexpr int kSoftmaxWarp0 = kIssuer0 + kIssuers;  // first softmax warp
  static constexpr int kThreads = 32 * kSoftmaxWarp0 + 128 * NT;
  static constexpr uint32_t kTmemCols = 512;
};

template <int NT>
struct __align__(1024) Smem {
  static constexpr int NS = Cfg<NT>::NS, KVH = Cfg<NT>::kKvHalf;
  uint8_t q[NT][2][kQHalf];    // [query tile][half of d][query][128 B]
  uint8_t k[NS][2][KVH];       // [stage][half of d][slot][128 B]
  uint8_t v[NS][2][KVH];       // [stage][half of d][slot][128 B]
  uint64_t q_full;
  uint64_t k_full[NS], v_full[NS], kv_empty[NS];
  uint64_t s_full[NT][2], p_full[NT][2];  // per (query tile, score buffer)
  uint64_t o_done[NT][2];  // P.V of tile j done, per (query tile, j & 1)
  uint64_t mma_done[NT];
  uint64_t tail_zero;  // the last tile's V rows past the visible end are zeroed
  uint32_t tmem_base;
};

// TMEM columns: score buffer b of query tile t at (2t + b) BN (the softmax
// stores P over its first BN/2 columns); O of query tile t at 256 + 128t.
template <int BN>
__device__ __forceinline__ uint32_t s_col(int t, int b) { return uint32_t(BN) * (2 * t + b); }
__device__ __forceinline__ uint32_t o_col(int t) { return 256u + 128u * t; }

__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float* f) {
  uint32_t r[128];
  asm volatile(PIE_TMEM_LD128_ASM : PIE_TMEM_LD_OUTS : "r"(taddr) : "memory");
#pragma unroll
  for (int i = 0; i < 128; ++i) f[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float* f) {
  uint32_t r[64];
  asm volatile(PIE_TMEM_LD64_ASM : PIE_TMEM_LD64_OUTS : "r"(taddr) : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) f[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st128(uint32_t taddr, const float* f) {
  uint32_t r[128];
#pragma unroll
  for (int i = 0; i < 128; ++i) r[i] = __float_as_uint(f[i]);
  asm volatile(PIE_TMEM_ST128_ASM ::"r"(taddr), PIE_TMEM_ST_INS : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(PIE_TMEM_ST32_ASM ::"r"(taddr), PIE_TMEM_ST32_INS : "memory");
}

__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t* r) {
  asm volatile(PIE_TMEM_ST64_ASM ::"r"(taddr), PIE_TMEM_ST64_INS : "memory");
}

// BN fp32 scores of this thread's TMEM lane, and BN/2 packed bf16 pairs back
template <int BN>
__device__ __forceinline__ void load_scores(uint32_t taddr, float* f) {
  if constexpr (BN == 128) tmem_ld128(taddr, f);
  else tmem_ld64(taddr, f);
}
template <int BN>
__device__ __forceinline__ void store_p(uint32_t taddr, const uint32_t* r) {
  if constexpr (BN == 128) tmem_st64(taddr, r);
  else tmem_st32(taddr, r);
}

}  // namespace tc

template <int NT>
__global__ void __launch_bounds__(tc::Cfg<NT>::kThreads, 1) attend_tc_kernel(
    DevMeta m, int G, int Hq, int Hkv, int P, float scale_log2,
    const uint32_t* mask_words, tc::Out out, uint32_t* status,
    const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
    const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap kgmap,
    const __grid_constant__ CUtensorMap vgmap) {
  using namespace tc;
  constexpr int NS = Cfg<NT>::NS, BN = Cfg<NT>::BN, kKvHalf = Cfg<NT>::kKvHalf;
  constexpr int D = 128;
  constexpr float kLn2 = 0.6931471805599453f;
  using SM = Smem<NT>;
  extern __shared__ uint8_t smem_raw[];
  SM& S = *reinterpret_cast<SM*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const TcItem it = m.tc_items[blockIdx.x];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the item is the plan's; everything below may be the kernels' before
  // (mask lists and counts, the queries, K/V scattered this pass)
  grid_dep_wait();
  // gather mode (masked passes): positions [kb, ke) of the row block's
  // compacted visible-slot list, this item's share of its tiles; otherwise
  // slots [kb, ke) of the lane
  const bool gather = it.block >= 0;
  int kb = it.kv_begin, ke = it.kv_end;
  MaskBlock mb{0, 0, 0, 0, 0, 0, 0, 0};
  if (gather) {
    mb = m.mblocks[it.block];
    const int U = m.list_len[it.block];
    const int tiles = (U + BN - 1) / BN;
    // the chunks this unit uses now that its list length is known; the
    // provisioned items past them have nothing to do and write nothing
    const int nch = masked_chunks(tiles, it.nchunks, *m.mask_tiles, Hkv, m.num_sms);
    if (it.chunk >= nch) return;
    kb = (it.chunk * tiles / nch) * BN;
    ke = min(U, ((it.chunk + 1) * tiles / nch) * BN);
  }
  const int T = ke > kb ? (ke - kb + BN - 1) / BN : 0;
  const int nqv = it.nrows * G;  // valid query vectors of the item
  // a page-granular list (whole pages, in list order) loads like the lane's
  // own pages; a slot-granular one is gathered row by row
  const bool page_list = gather && m.list_mode[it.block] != 0;
  const bool row_gather = gather && !page_list;

  if (threadIdx.x == 0) {
    mbar_init(&S.q_full, 1);
    for (int t = 0; t < NT; ++t) mbar_init(&S.mma_done[t], 1);
    mbar_init(&S.tail_zero, 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(&S.k_full[i], 1);
      mbar_init(&S.v_full[i], 1);
      mbar_init(&S.kv_empty[i], Cfg<NT>::kIssuers);  // released by every issuer's P.V
    }
    for (int t = 0; t < NT; ++t) {
      for (int b = 0; b < 2; ++b) {
        mbar_init(&S.s_full[t][b], 1);
        mbar_init(&S.p_full[t][b], 4);
      }
      mbar_init(&S.o_done[t][0], 1);
      mbar_init(&S.o_done[t][1], 1);
    }
    fence_barrier_init();
  }
  if (warp == Cfg<NT>::kIssuer0 && T > 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&S.tmem_base)),
                 "r"(Cfg<NT>::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = S.tmem_base;
  bool bad = false;
  grid_dep_launch();  // the combine kernel may start (it waits for this one)

  if (warp < Cfg<NT>::kIssuer0) {
    // ---------------- TMA producers: warp 0 loads K, warp 1 loads V ----------
    // A warp's TMA copies issue one after another, so every copy of a tile
    // comes from its own lane and the two tensors from two warps.
    //   pages (the lane's own, or a page-granular list):
    //                lane 2i + a -> page (ts / P + i) of the tile, half a of d
    //                (at most BN / P <= 16 pages)
    //   row gather:  lane o (and o + 32 for 128-slot tiles) -> rows 4(o/2) ..
    //                4(o/2) + 3 of the tile, half o % 2 of d, one gather4 each
    // The copies' pool rows come from the page table or the pool rows of the
    // listed slots, fetched one tile ahead.
    const bool is_v = warp == 1;
    if (T > 0) {
      const uint64_t pol = policy_evict_first();
      if (!is_v && lane == 0) {
        mbar_arrive_expect_tx(&S.q_full, NT * 2 * kQHalf);
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
          for (int a = 0; a < 2; ++a)
            tma_4d(S.q[t][a], &qmap, 64 * a, 0, it.kv_head, it.row0 + t * (kTcTileQueries / G),
                   &S.q_full);
      }
      const CUtensorMap* map = row_gather ? (is_v ? &vgmap : &kgmap) : (is_v ? &vmap : &kmap);
      uint64_t* full = is_v ? S.v_full : S.k_full;
      const int32_t* pages = m.page_ids + m.page_indptr[it.lane];
      const int32_t* lrow = gather ? m.lrow + mb.list_off : nullptr;
      const int hrow = it.kv_head * P;  // row offset of this kv head within a page
      constexpr int GOPS = BN / 64;     // gather4 copies per lane and tile
      int y[GOPS][4];
      auto coords = [&](int jj) {
        const int ts = kb + jj * BN;
        const int te = min(ts + BN, ke);
        if (row_gather) {
          const int rows = ((te - ts) + 15) & ~15;
#pragma unroll
          for (int i = 0; i < GOPS; ++i) {
            const int r0 = 4 * ((lane + 32 * i) >> 1);
            if (r0 < rows) {
              // rows past the last listed slot repeat it (finite data for
              // the zero-weight columns of the last 16-slot MMA step)
#pragma unroll
              for (int e = 0; e < 4; ++e) y[i][e] = lrow[min(ts + r0 + e, te - 1)] + hrow;
            }
          }
        } else {
          const int p0 = ts / P, p1 = (te - 1) / P;
          if ((lane >> 1) <= p1 - p0)
            y[0][0] = page_list ? lrow[ts + (lane >> 1) * P] + hrow
                                : (pages[p0 + (lane >> 1)] * Hkv + it.kv_head) * P;
        }
      };
      coords(0);
      for (int j = 0; j < T; ++j) {
        const int st = j % NS;
        if (j >= NS && !mbar_wait(&S.kv_empty[st], ((j / NS) - 1) & 1)) {
          bad = true;
          break;
        }
        const int ts = kb + j * BN;
        const int te = min(ts + BN, ke);
        uint8_t* dst = is_v ? S.v[st][0] : S.k[st][0];  // half a at + a * kKvHalf
        if (row_gather) {
          const int rows = ((te - ts) + 15) & ~15;
          if (lane == 0) mbar_arrive_expect_tx(&full[st], uint32_t(rows) * 128u * 2u);
          __syncwarp();
#pragma unroll
          for (int i = 0; i < GOPS; ++i) {
            const int o = lane + 32 * i, a = o & 1, r0 = 4 * (o >> 1);
            if (r0 < rows)
              tma_gather4(dst + a * kKvHalf + r0 * 128, map, 64 * a, y[i][0], y[i][1], y[i][2],
                          y[i][3], &full[st], pol);
          }
        } else {
          const int p0 = ts / P, p1 = (te - 1) / P;
          if (lane == 0) mbar_arrive_expect_tx(&full[st], uint32_t(p1 - p0 + 1) * P * 128u * 2u);
          __syncwarp();
          const int pg = lane >> 1, a = lane & 1;
          if (pg <= p1 - p0)
            tma_2d(dst + a * kKvHalf + ((p0 + pg) * P - ts) * 128, map, 64 * a, y[0][0], &full[st],
                   pol);
        }
        if (j + 1 < T) coords(j + 1);
      }
      if (is_v) {
        // The last tile's V rows between its last visible slot and the end of
        // that 16-slot MMA step hold whatever the page held past kv_len: once
        // the tile has landed they are zeroed here, before any issuer's last
        // P.V (which waits on tail_zero).  Row gathers load finite rows there.
        const int tl = kb + (T - 1) * BN, vl = min(BN, ke - tl);
        if (!row_gather && (vl & 15) && !bad) {
          const int stl = (T - 1) % NS;
          if (mbar_wait(&S.v_full[stl], ((T - 1) / NS) & 1)) {
            const int nr = ((vl + 15) & ~15) - vl;
            for (int i = lane; i < nr * 16; i += 32) {
              const int h = i / (nr * 8), rem = i % (nr * 8);
              *reinterpret_cast<uint4*>(S.v[stl][h] + (vl + rem / 8) * 128 + (rem % 8) * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
          } else {
            bad = true;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.tail_zero);
      }
    }
  } else if (warp < Cfg<NT>::kSoftmaxWarp0) {
    // ---------------- MMA issuers: one warp per query tile ---------------------
    // Each issuer keeps its own tile's chain (S, softmax, P.V, next S) in
    // flight, so one tile's handoff waits overlap the other's MMAs in the
    // shared tensor pipe.  Shared-memory descriptors are built once and
    // advanced by constant increments (address field in 16-byte units).
    if (lane == 0 && T > 0) {
      const int t = warp - Cfg<NT>::kIssuer0;
      constexpr uint32_t ID_S = idesc(128, BN, false);
      constexpr uint32_t ID_O = idesc(128, 128, true);
      const uint64_t dq = sdesc(S.q[t][0], 16, 1024);              // + (kQHalf >> 4) per half
      const uint64_t dk = sdesc(S.k[0][0], 16, 1024);              // + (2 kKvHalf >> 4) per stage
      const uint64_t dv = sdesc(S.v[0][0], kKvHalf, 1024);         // + 128 per 16-slot step
      const uint32_t tO = tmem + o_col(t);
      // S_t(j) = Q_t K_j^T into score buffer j & 1
      auto issue_s = [&](int j) -> bool {
        const int st = j % NS;
        if (!mbar_wait(&S.k_full[st], (j / NS) & 1)) return false;
        fence_after();
        const uint32_t d = tmem + s_col<BN>(t, j & 1);
        const uint64_t bk = dk + uint64_t(st) * (2 * kKvHalf >> 4);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t off = uint64_t((k >> 2) * (kQHalf >> 4) + (k & 3) * 2);
          const uint64_t offk = uint64_t((k >> 2) * (kKvHalf >> 4) + (k & 3) * 2);
          mma_ss(d, dq + off, bk + offk, ID_S, k > 0 ? 1u : 0u);
        }
        commit(&S.s_full[t][j & 1]);
        return true;
      };
      // O_t += P_t(j) V_j once the softmax group has stored P_t(j)
      auto issue_pv = [&](int j) -> bool {
        if (!mbar_wait(&S.p_full[t][j & 1], (j >> 1) & 1)) return false;
        const int st = j % NS;
        if (!mbar_wait(&S.v_full[st], (j / NS) & 1)) return false;
        if (j == T - 1 && !mbar_wait(&S.tail_zero, 0)) return false;
        fence_after();
        const int valid = min(BN, ke - (kb + j * BN));
        const int ksteps = (valid + 15) >> 4;
        const uint64_t bv = dv + uint64_t(st) * (2 * kKvHalf >> 4);
        const uint32_t ta = tmem + s_col<BN>(t, j & 1);
        for (int k = 0; k < ksteps; ++k)
          mma_ts(tO, ta + 8 * k, bv + uint64_t(k) * (2048 >> 4), ID_O, (j > 0 || k > 0) ? 1u : 0u);
        commit(&S.o_done[t][j & 1]);
        commit(&S.kv_empty[st]);
        return true;
      };
      bool ok = mbar_wait(&S.q_full, 0);
      for (int jj = 0; jj < 2 && jj < T && ok; ++jj) ok = issue_s(jj);
      for (int j = 0; j < T && ok; ++j) {
        ok = issue_pv(j);
        if (ok && j + 2 < T) ok = issue_s(j + 2);
      }
      // every MMA of this issuer must have finished before TMEM is released
      commit(&S.mma_done[t]);
      if (!mbar_wait(&S.mma_done[t], 0)) ok = false;
      bad = !ok;
    }
  } else if (T > 0) {
    // ---------------- softmax groups: thread = query row ---------------------
    const int t = (warp - Cfg<NT>::kSoftmaxWarp0) >> 2;  // query tile of this group
    const int quad = warp & 3;          // TMEM lane quadrant of this warp
    const int qm = quad * 32 + lane;    // query row within the tile == TMEM lane
    const int q = t * kTcTileQueries + qm;
    const bool valid_q = q < nqv;
    const bool warp_live = __any_sync(0xffffffffu, valid_q);
    const int row = it.row0 + (valid_q ? q : 0) / G;
    const int head = it.kv_head * G + (valid_q ? q : 0) % G;
    const int row_slot = valid_q ? m.slots[row] : INT_MAX;
    // the row's mask words: over the compacted list (gather mode) or over
    // the lane's slots; nullptr without a mask
    const bool masked = mask_words != nullptr;
    const uint32_t* mrow = nullptr;
    if (masked && valid_q)
      mrow = gather ? m.cmask + mb.cmask_off + int64_t(row - mb.r0) * mb.nw
                    : mask_words + m.mask_word_indptr[row];
    const uint32_t lane_base = tmem + (uint32_t(quad * 32) << 16);
    const uint32_t tO = lane_base + o_col(t);
    float m_used = -INFINITY, l_run = 0.f;
    // the row's mask words of the next tile are loaded one tile ahead
    constexpr int NW = BN / 32;  // mask words per tile
    uint32_t wnext[NW];
    auto load_words = [&](int jj) {
      const int tt = kb + jj * BN;
#pragma unroll
      for (int i = 0; i < NW; ++i) wnext[i] = !mrow ? ~0u : (tt + 32 * i < ke ? mrow[(tt >> 5) + i] : 0u);
    };
    load_words(0);
    for (int j = 0; j < T; ++j) {
      const int ts = kb + j * BN;
      const uint32_t tS = lane_base + s_col<BN>(t, j & 1);
      uint32_t words[NW];
#pragma unroll
      for (int i = 0; i < NW; ++i) words[i] = wnext[i];
      if (j + 1 < T) load_words(j + 1);
      if (!mbar_wait(&S.s_full[t][j & 1], (j >> 1) & 1)) { bad = true; break; }
      fence_after();
      if (warp_live) {
        float s[BN];
        load_scores<BN>(tS, s);
        // a tile every column of which every live row of the warp sees
        uint32_t wand = ~0u;
#pragma unroll
        for (int i = 0; i < NW; ++i) wand &= words[i];
        const bool all_vis = (ts + BN <= ke) &&
                             (masked ? (wand == ~0u) : (ts + BN - 1 <= row_slot));
        if (!__all_sync(0xffffffffu, all_vis || !valid_q)) {
#pragma unroll
          for (int c = 0; c < BN; ++c) {
            const int sa = ts + c;
            const bool vis = valid_q && sa < ke &&
                             (masked ? ((words[c >> 5] >> (c & 31)) & 1u) != 0 : sa <= row_slot);
            s[c] = vis ? s[c] : -INFINITY;
          }
        }
        // row max: three-input max over four independent chains
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < BN; c += 8) {
#pragma unroll
          for (int i = 0; i < 4; ++i) m4[i] = max3(m4[i], s[c + 2 * i], s[c + 2 * i + 1]);
        }
        const float mx = max3(m4[0], m4[1], fmaxf(m4[2], m4[3]));
        const float m_tile = mx * scale_log2;  // scale > 0: max commutes with it
        float m_new = m_used;
        if (m_used == -INFINITY || m_tile > m_used + 8.f) m_new = fmaxf(m_used, m_tile);
        const float alpha = (m_new == m_used) ? 1.f : ex2(m_used - m_new);
        const float neg_m = (m_new == -INFINITY) ? 0.f : -m_new;
        // p = 2^(s * scale - m) for a pair per packed FMA; row sum by packed
        // adds into four pair accumulators
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        uint32_t pk[BN / 2];
#pragma unroll
        for (int c = 0; c < BN / 2; ++c) {
          float x0, x1;
          ffma2(x0, x1, s[2 * c], s[2 * c + 1], scale_log2, scale_log2, neg_m, neg_m);
          const float p0 = ex2(x0), p1 = ex2(x1);
          fadd2(acc[2 * (c & 3)], acc[2 * (c & 3) + 1], p0, p1);
          __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
          pk[c] = *reinterpret_cast<uint32_t*>(&h2);
        }
        fadd2(acc[0], acc[1], acc[2], acc[3]);
        fadd2(acc[4], acc[5], acc[6], acc[7]);
        fadd2(acc[0], acc[1], acc[4], acc[5]);
        l_run = l_run * alpha + (acc[0] + acc[1]);
        m_used = m_new;
        // The buffer's previous P was read by P.V of tile j-2, which the
        // tensor pipe executed before this tile's S, so P may be stored now.
        store_p<BN>(tS, pk);
        // O is rescaled, by the warps whose rows need it, only after P.V of
        // tile j-1 has landed in it.  The completion barriers of P.V form a
        // ring of two (by j & 1): P.V of tile j+1 cannot complete before this
        // group arrives on p_full for it, so a warp that skips waits never
        // sees a barrier two phases ahead of the one it waits on.
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          if (!mbar_wait(&S.o_done[t][(j - 1) & 1], ((j - 1) >> 1) & 1)) { bad = true; break; }
          fence_after();
          float o[128];
          tmem_ld128(tO, o);
#pragma unroll
          for (int c = 0; c < 128; ++c) o[c] *= alpha;
          tmem_st128(tO, o);
        }
      }
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.p_full[t][j & 1]);
    }
    if (warp_live && !bad) {
      if (!mbar_wait(&S.o_done[t][(T - 1) & 1], ((T - 1) >> 1) & 1)) {
        bad = true;
      } else {
        fence_after();
        float o[128];
        tmem_ld128(tO, o);
        if (valid_q) {
          if (it.direct) {
            const bool empty = !(l_run > 0.f);
            const float inv = empty ? 0.f : 1.f / l_run;
            const float lse = empty ? -INFINITY : (m_used + log2f(l_run)) * kLn2;
            uint4 packed[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                __nv_bfloat162 h2 =
                    __floats2bfloat162_rn(o[8 * c + 2 * e] * inv, o[8 * c + 2 * e + 1] * inv);
                w[e] = *reinterpret_cast<uint32_t*>(&h2);
              }
              packed[c] = make_uint4(w[0], w[1], w[2], w[3]);
            }
            write_row(m, out, Hq, row, head, packed, lse);
          } else {
            float4* po = reinterpret_cast<float4*>(m.part_o + int64_t(it.part_base + q) * D);
#pragma unroll
            for (int c = 0; c < 32; ++c)
              po[c] = make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
            m.part_ml[it.part_base + q] = make_float2(m_used, l_run);
          }
        }
      }
    }
  }
  if (T == 0 && threadIdx.x < NT * 128) {
    // nothing visible in this chunk: an empty partial state (a direct item
    // with no visible slot writes zeros and -inf)
    const int q = threadIdx.x;
    if (q < nqv) {
      if (it.direct) {
        uint4 zero[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) zero[c] = make_uint4(0u, 0u, 0u, 0u);
        write_row(m, out, Hq, it.row0 + q / G, it.kv_head * G + q % G, zero, -INFINITY);
      } else {
        float* po = m.part_o + int64_t(it.part_base + q) * D;
        for (int c = 0; c < D; ++c) po[c] = 0.f;
        m.part_ml[it.part_base + q] = make_float2(-INFINITY, 0.f);
      }
    }
  }
  if (bad) set_status(status, PIE_STATUS_TIMEOUT);
  fence_before();
  __syncthreads();
  if (warp == Cfg<NT>::kIssuer0 && T > 0) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(Cfg<NT>::kTmemCols)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------
// host side: tensor maps and launch
// ---------------------------------------------------------------------------
template <int NT>
static cudaError_t launch_nt(const pie_fwd_plan_t& p, const uint32_t* mask_words, tc::Out out,
                             uint32_t* status, const CUtensorMap& qm, const CUtensorMap& km,
                             const CUtensorMap& vm, const CUtensorMap& kgm,
                             const CUtensorMap& vgm, cudaStream_t s) {
  const size_t smem = sizeof(tc::Smem<NT>) + 1024;
  static std::atomic<uint64_t> configured{0};
  cudaError_t e = set_smem_limit(attend_tc_kernel<NT>, int(smem), configured);
  if (e != cudaSuccess) return e;
  return launch_dependent(attend_tc_kernel<NT>, dim3(p.num_tc_items), dim3(tc::Cfg<NT>::kThreads),
                          smem, s, true, p.dev, p.G, p.desc.num_q_heads, p.desc.num_kv_heads,
                          p.desc.page_size, p.desc.sm_scale * 1.4426950408889634f, mask_words, out,
                          status, qm, km, vm, kgm, vgm);
}

cudaError_t launch_attend_tc(const pie_fwd_plan_t& p, const void* q_rot, const void* k_pool,
                             const void* v_pool, const uint32_t* mask_words, void* out_readout,
                             float* lse_readout, void* out_all, float* lse_all, uint32_t* status,
                             cudaStream_t s) {
  const int D = p.desc.head_dim, Hq = p.desc.num_q_heads, Hkv = p.desc.num_kv_heads;
  const int G = p.G, P = p.desc.page_size;
  if (D != 128 || p.desc.dtype != PIE_BF16 || kTcTileQueries % G != 0) return cudaErrorNotSupported;
  CUtensorMap qm, km, vm;
  {
    const cuuint64_t dims[4] = {cuuint64_t(D), cuuint64_t(G), cuuint64_t(Hkv), cuuint64_t(p.N)};
    const cuuint64_t str[3] = {cuuint64_t(D) * 2, cuuint64_t(G) * D * 2, cuuint64_t(Hq) * D * 2};
    const cuuint32_t box[4] = {64, cuuint32_t(G), 1, cuuint32_t(kTcTileQueries / G)};
    if (!tc::make_map(&qm, q_rot, 4, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {cuuint64_t(D), cuuint64_t(p.num_pool_pages) * Hkv * P};
    const cuuint64_t str[1] = {cuuint64_t(D) * 2};
    const cuuint32_t box[2] = {64, cuuint32_t(P)};
    if (!tc::make_map(&km, k_pool, 2, dims, str, box)) return cudaErrorInvalidValue;
    if (!tc::make_map(&vm, v_pool, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  // one-row boxes for the slot-granular gathers of masked passes
  CUtensorMap kgm = km, vgm = vm;
  if (p.num_mblocks > 0) {
    const cuuint64_t dims[2] = {cuuint64_t(D), cuuint64_t(p.num_pool_pages) * Hkv * P};
    const cuuint64_t str[1] = {cuuint64_t(D) * 2};
    const cuuint32_t box[2] = {64, 1};
    if (!tc::make_map(&kgm, k_pool, 2, dims, str, box)) return cudaErrorInvalidValue;
    if (!tc::make_map(&vgm, v_pool, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  tc::Out out{static_cast<__nv_bfloat16*>(out_readout), lse_readout,
              static_cast<__nv_bfloat16*>(out_all), lse_all};
  return p.tc_nt == 2 ? launch_nt<2>(p, mask_words, out, status, qm, km, vm, kgm, vgm, s)
                      : launch_nt<1>(p, mask_words, out, status, qm, km, vm, kgm, vgm, s);
}

}  // namespace pie
