// Step 2-3 of a ForwardPass for lanes with few query vectors per kv head
// (decode rows, short drafts), bf16 K/V with head_dim 128: split-KV grouped-
// query attention over paged K/V (Pie "The forward pass": State geometry
// kv_len; Attention masks), with the dot products and the probability-
// weighted sums on the tensor cores' warp-level MMA.
//
// The pass is bound by HBM: every visible slot's K and V head rows are read
// once for the NQ (2, 4 or 8) query vectors of a GQA group.  Computing those
// few dot products with scalar FMAs costs about 57 warp instructions per
// (slot, kv head), enough to keep the kernel short of the copy bandwidth, so
// here each compute warp takes its 16 slots of a 64-slot stage with 16 x 8
// x 16 bf16 MMAs, both products transposed so that the (up to 8) query
// vectors are the MMA's 8 columns and no row is padding:
//   * S^T = K Q^T: eight MMAs over d, K fragments read with ldmatrix;
//   * the online softmax on the accumulator fragments: each query's 16
//     scores sit in the 8 lanes of its column (three shuffles for the
//     maximum), and the running maximum used for the exponent only moves
//     when a unit's maximum exceeds it by more than 2^8, so the output is
//     rarely rescaled;
//   * O^T += V^T P^T: eight MMAs, one per 16-wide tile of d, V fragments read
//     with ldmatrix.trans; the probabilities (bf16) become the B operand by
//     an in-register 8 x 8 transpose (movmatrix) of the score fragments.
// That is about 60 warp instructions per warp and stage where the scalar
// kernel needs about 900.  The fragments need K and V rows in shared memory
// without bank conflicts between slots, so the producer warp copies each
// (page, kv head) block as two 2-D tensor boxes of P rows x 128 bytes (one
// per half of d) with the 128-byte swizzle; with three CTAs per SM, each with
// a two-stage ring, those copies stream at the copy bandwidth.
// In a masked pass an item walks its chunk of the compacted list of the slots
// its rows see (Attention masks; built by the mask pre-pass): the producer
// copies the listed whole pages of a window-like list the same way, or the
// listed rows of a scattered list four at a time (tile::gather4 over one-row
// boxes), and the rows' visibility comes from their mask words re-expressed
// over the list.
// Each work item writes one partial (max, sum, unnormalised output) per query
// vector; the combine kernel (combine.cu) merges an item's chunks.  Every wait
// is bounded in time.

#include "common.cuh"
#include "tc_util.cuh"

namespace pie {

namespace dm {

constexpr int D = 128;
constexpr int WARPS = 4;                           // compute warps (+1 producer warp)
constexpr int THREADS = (WARPS + 1) * 32;
constexpr int HALF_BYTES = kStageSlots * 128;      // one half of d of a stage's K (or V): 8 KB
constexpr int STAGE_BYTES = 4 * HALF_BYTES;        // K halves, then V halves: 32 KB
constexpr int STAGES = 2;                          // a 64 KB ring: three CTAs per SM
constexpr int Q_BYTES = 8 * D * 2;                 // the item's query vectors (8 rows), swizzled
constexpr int SMEM = STAGES * STAGE_BYTES + Q_BYTES + 1024 + 2 * STAGES * 8 + 64;  // + align,
                                                                           // barriers, item queue
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D (16 x 8, fp32) += A (16 x 16, bf16) B (16 x 8, bf16), fragments in the
// warp-level MMA layout
__device__ __forceinline__ void mma16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// the transpose of an 8 x 8 matrix of 16-bit elements held one pair per lane
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// shared-memory address of 16-byte chunk c (0..15 over d) of stage row r in
// a half-split, 128-byte-swizzled K or V block starting at base
__device__ __forceinline__ uint32_t chunk_addr(uint32_t base, int r, int c) {
  return base + uint32_t((c >> 3) * HALF_BYTES + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

}  // namespace dm

// One work item as the kernel walks it: slots (or list positions) [kb, ke).
struct DecRange {
  DecItem it;
  MaskBlock mb;
  int kb, ke, nstages;
  bool listed, page_list, skip;  // skip: a listed chunk past the list's share
};

template <int NQ>
__global__ void __launch_bounds__(dm::THREADS, 3) attend_decode_mma_kernel(
    DevMeta m, int Hq, int Hkv, int G, int P, float scale_log2, const __nv_bfloat16* q_rot,
    const uint32_t* mask_words, int list_tile, int num_items, int items_per_cta,
    uint32_t* status, const __grid_constant__ CUtensorMap kmap,
    const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap kgmap,
    const __grid_constant__ CUtensorMap vgmap) {
  using namespace dm;
  static_assert(NQ <= 8, "query vectors of an item fill at most the 8 MMA columns");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* qs = ring + STAGES * STAGE_BYTES;  // query vector q, 16-byte chunk c at q * 256 + (c ^ q) * 16
  uint64_t* full = reinterpret_cast<uint64_t*>(qs + Q_BYTES);
  uint64_t* empty = full + STAGES;
  // item queue: the producer hands each item index (or -1: no more) to the
  // compute warps through two slots; compute warp 0 reads a slot and writes
  // the decision every compute warp then takes (-2: the wait ran out)
  uint64_t* item_full = empty + STAGES;
  uint64_t* item_empty = item_full + 2;
  int* qidx = reinterpret_cast<int*>(item_empty + 2);
  int* decision = qidx + 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], WARPS);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(&item_full[q], 1);
      mbar_init(&item_empty[q], 1);
    }
    fence_barrier_init();
  }
  __syncthreads();
  // everything below, the work items included, is read after the wait (the
  // items may come from a kernel queued just before this one)
  grid_dep_wait();
  grid_dep_launch();
  // This CTA's items: taken one by one from the plan's work counter (a
  // persistent grid), or, without a counter, items_per_cta consecutive ones.
  // The producer runs its stages straight through from one item into the
  // next (the ring's stages and phases continue), so the next item's first
  // copies are in flight while the compute warps merge the last one.
  int* const work = m.dec_work;
  const int first = blockIdx.x * items_per_cta;
  const int last = min(num_items, first + items_per_cta);
  auto resolve = [&](int idx) {
    DecRange r;
    r.it = m.dec_items[idx];
    r.kb = r.it.kv_begin;
    r.ke = r.it.kv_end;
    // a listed item: chunk kv_begin of the kv_end provisioned ones of its
    // block's list, in whole list tiles (the split the combine step computes
    // the same way); chunks past the list's share write nothing
    r.listed = r.it.block >= 0;
    r.page_list = false;
    r.skip = false;
    r.mb = MaskBlock{0, 0, 0, 0, 0, 0, 0, 0};
    if (r.listed) {
      r.mb = m.mblocks[r.it.block];
      const int U = m.list_len[r.it.block];
      const int tiles = (U + list_tile - 1) / list_tile;
      const int nch =
          masked_chunks(tiles, r.it.kv_end, *m.mask_tiles, Hkv, m.num_sms * kDecListWaves);
      r.skip = r.it.kv_begin >= nch;
      r.kb = (r.it.kv_begin * tiles / max(nch, 1)) * list_tile;
      r.ke = min(U, ((r.it.kv_begin + 1) * tiles / max(nch, 1)) * list_tile);
      r.page_list = m.list_mode[r.it.block] != 0;
    }
    r.nstages = (!r.skip && r.ke > r.kb) ? (r.ke - r.kb + kStageSlots - 1) / kStageSlots : 0;
    return r;
  };
  const uint64_t wait_ns = m.test_wait_us ? uint64_t(m.test_wait_us) * 1000ull : kWaitLimitNs;

  if (warp == WARPS) {
    // ---------------- producer warp: 2-D tensor copies of K/V pages -----------
    // Whole pages (the lane's own, or the listed pages of a window-like list,
    // page i of the list at positions i * P ..): lane 4i + c copies block c
    // (K half 0, K half 1, V half 0, V half 1) of page (stage start / P + i); a
    // stage spans 64 / P pages (at most 8), and the page ids of the next stage
    // are fetched while this one is issued.  A scattered list: lane i gathers
    // rows 4(i % 16) .. 4(i % 16) + 3 of every stage from K (i < 16) or V, both
    // halves of d; rows past the last listed one repeat it (finite data, never
    // visible).  A page id outside the pool is not copied and sets
    // PIE_STATUS_BOUNDS.
    const uint64_t pol = policy_evict_first();
    const int c = lane & 3, pi = lane >> 2;
    const int gi = lane & 15, tv = lane >> 4;
    int gs = 0;  // stages issued by this CTA so far (ring slot gs % STAGES)
    // every way out of the producer counts the CTA done; the last CTA done
    // sets the counter back to zero for the next launch
    auto finish = [&]() {
      if (work && lane == 0) {
        __threadfence();
        if (atomicAdd(work + 1, 1) == int(gridDim.x) - 1) {
          atomicExch(work, 0);
          atomicExch(work + 1, 0);
        }
      }
    };
    for (int k = 0;; ++k) {
      // the next item: from the counter, or the CTA's next fixed one
      int idx;
      if (work) {
        idx = 0;
        if (lane == 0) idx = atomicAdd(work, 1);
        idx = __shfl_sync(0xffffffffu, idx, 0);
        if (idx >= num_items) idx = -1;
      } else {
        idx = first + k < last ? first + k : -1;
      }
      const int q = k & 1;
      if (k >= 2 && !mbar_wait_ns(&item_empty[q], ((k >> 1) - 1) & 1, wait_ns)) {
        if (lane == 0) set_status(status, PIE_STATUS_TIMEOUT);
        finish();
        return;
      }
      if (lane == 0) {
        qidx[q] = idx;
        mbar_arrive(&item_full[q]);  // release: the index is visible to the waiters
      }
      if (idx < 0) break;
      const DecRange r = resolve(idx);
      const int32_t* pages = m.page_ids + m.page_indptr[r.it.lane];
      // a listed slot's row in the pools viewed as [rows][d], less kv_head * P
      const int32_t* lrow = r.listed ? m.lrow + r.mb.list_off : nullptr;
      const bool gather = r.listed && !r.page_list;
      const int hrow = r.it.kv_head * P;
      auto page_of = [&](int s) -> int64_t {
        const int sb = r.kb + s * kStageSlots;
        const int p0 = sb / P, p1 = (min(sb + kStageSlots, r.ke) - 1) / P;
        if (pi > p1 - p0) return 0;
        return r.listed ? int64_t(lrow[(p0 + pi) * P]) / (int64_t(Hkv) * P)
                        : int64_t(pages[p0 + pi]);
      };
      int64_t pid = (r.nstages > 0 && !gather) ? page_of(0) : 0;
      for (int s = 0; s < r.nstages; ++s, ++gs) {
        // test hook: stop before this stage of the first item (no copy of it,
        // or of anything later, is ever issued)
        if (s == m.test_stall - 1) {
          finish();
          return;
        }
        const int st = gs % STAGES, use = gs / STAGES;
        if (use > 0 && !mbar_wait_ns(&empty[st], (use - 1) & 1, wait_ns)) {
          if (lane == 0) set_status(status, PIE_STATUS_TIMEOUT);
          finish();
          return;
        }
        const int sb = r.kb + s * kStageSlots;
        if (gather) {
          const int n = min(kStageSlots, r.ke - sb);
          const int ng = (n + 3) >> 2;
          if (lane == 0) mbar_arrive_expect_tx(&full[st], uint32_t(ng) * 4u * 128u * 2u * 2u);
          __syncwarp();
          if (gi < ng) {
            int y[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) y[e] = lrow[sb + min(4 * gi + e, n - 1)] + hrow;
            uint8_t* dst = ring + st * STAGE_BYTES + tv * 2 * HALF_BYTES + 4 * gi * 128;
#pragma unroll
            for (int a = 0; a < 2; ++a)
              tc::tma_gather4(dst + a * HALF_BYTES, tv ? &vgmap : &kgmap, 64 * a, y[0], y[1],
                              y[2], y[3], &full[st], pol);
          }
          continue;
        }
        const int se = min(sb + kStageSlots, r.ke);
        const int p0 = sb / P, p1 = (se - 1) / P;
        const bool mine = pi <= p1 - p0;
        const bool in_pool = pid >= 0 && pid < m.num_pool_pages;
        const bool issue = mine && in_pool;
        const uint32_t copies = __popc(__ballot_sync(0xffffffffu, issue));
        if (lane == 0) {
          if (copies != 4u * uint32_t(p1 - p0 + 1)) set_status(status, PIE_STATUS_BOUNDS);
          mbar_arrive_expect_tx(&full[st], copies * uint32_t(P) * 128u);
        }
        __syncwarp();
        if (issue) {
          uint8_t* dst = ring + st * STAGE_BYTES + (c >> 1) * 2 * HALF_BYTES +
                         (c & 1) * HALF_BYTES + ((p0 + pi) * P - sb) * 128;
          tc::tma_2d(dst, (c >> 1) ? &vmap : &kmap, 64 * (c & 1), int((pid * Hkv + r.it.kv_head) * P),
                     &full[st], pol);
        }
        if (s + 1 < r.nstages) pid = page_of(s + 1);
      }
    }
    finish();
    return;
  }

  // ---------------- compute warps ---------------------------------------------
  // Fragments (g = lane / 4, t = lane % 4).  Both products are taken
  // transposed, so that the query vectors are the 8 columns of the MMA and no
  // row is padding:
  //   S^T (16 slots x 8 queries) = K (16 slots x 128 d) Q^T: lane holds
  //     S^T[slot g][q 2t, 2t+1] and S^T[slot g + 8][q 2t, 2t+1];
  //   O^T (16 d x 8 queries) += V^T (16 d x 16 slots) P^T, for each of the
  //     eight 16-wide tiles of d: lane holds O^T[d g][q 2t, 2t+1] and
  //     O^T[d g + 8][q 2t, 2t+1] of its tile.
  // So each lane keeps the online softmax of queries 2t and 2t + 1; a
  // query's 16 scores of a unit sit in the 8 lanes of its column pair.
  const int g = lane >> 2, t = lane & 3;
  const uint32_t ring_s = smem_u32(ring);
  const uint32_t qs_s = smem_u32(qs);
  // ldmatrix row addresses: lane i serves row i & 7 of matrix i >> 3
  const int mi = lane >> 3, mr = lane & 7;
  int gs = 0;  // stages consumed by this CTA so far
  // A warp whose wait for a stage runs out stops computing and arriving for
  // the rest of the CTA's items, but still takes every named barrier below
  // (the other warps' waits end too, bounded), so the CTA ends; the status
  // word says the outputs are not valid.
  bool dead = false;
  for (int k = 0;; ++k) {
    // the item the producer handed over, decided once for all compute warps
    if (warp == 0) {
      const int q = k & 1;
      const bool ok = mbar_wait_ns(&item_full[q], (k >> 1) & 1, wait_ns);
      int v = ok ? qidx[q] : -2;
      v = __shfl_sync(0xffffffffu, v, 0);
      if (lane == 0) {
        decision[k & 1] = v;
        if (v != -2) mbar_arrive(&item_empty[q]);
        if (v == -2) set_status(status, PIE_STATUS_TIMEOUT);
      }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(WARPS * 32) : "memory");
    const int idx = decision[k & 1];
    if (idx < 0) break;
    const DecRange r = resolve(idx);
    if (r.skip) continue;
    const DecItem& it = r.it;
    const int kb = r.kb, ke = r.ke, nstages = r.nstages;
    const int nqv = it.nrows * G;
    // the query vectors into shared memory (zeros past the item's), 16 bytes
    // per thread, chunks XOR-swizzled by the row so that ldmatrix reads of
    // the eight rows hit distinct banks; the B fragments of Q^T are read from
    // there at every stage (b0 = Q[g][16k + 2t, +1], b1 = Q[g][16k + 2t + 8, +9]).
    // The previous item's reads of them ended before its merge.
    {
      const int qv = threadIdx.x >> 4, ch = threadIdx.x & 15;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (qv < nqv) {
        const int row = it.row0 + qv / G, head = it.kv_head * G + qv % G;
        v = *reinterpret_cast<const uint4*>(q_rot + (int64_t(row) * Hq + head) * D + ch * 8);
      }
      *reinterpret_cast<uint4*>(qs + qv * 256 + ((ch ^ qv) << 4)) = v;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(WARPS * 32) : "memory");
    // this lane's two query vectors 2t + i: validity, causal limit, mask row
    bool valid_q[2];
    int slot_lim[2];
    const uint32_t* mrow[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int qv = 2 * t + i;
      valid_q[i] = qv < nqv;
      const int row = it.row0 + (valid_q[i] ? qv : 0) / G;
      slot_lim[i] = valid_q[i] ? m.slots[row] : -1;
      // mask words: the row's own over the lane's slots, or, for a listed
      // item, re-expressed over its block's list
      mrow[i] = !valid_q[i] ? nullptr
                : r.listed  ? m.cmask + r.mb.cmask_off + int64_t(row - r.mb.r0) * r.mb.nw
                : mask_words ? mask_words + m.mask_word_indptr[row]
                             : nullptr;
    }
    float o[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_used[2] = {-INFINITY, -INFINITY}, l_part[2] = {0.f, 0.f};
    // the rows' mask words of this warp's unit, fetched one stage ahead
    uint32_t wnext[2] = {~0u, ~0u};
    auto load_words = [&](int ss) {
      const int ub = kb + ss * kStageSlots + warp * kWarpSlots;
#pragma unroll
      for (int i = 0; i < 2; ++i)
        wnext[i] = (mrow[i] && ub < ke) ? (mrow[i][ub >> 5] >> (ub & 31)) : ~0u;
    };
    if (nstages > 0) load_words(0);

    for (int s = 0; s < nstages; ++s, ++gs) {
      const int st = gs % STAGES;
      const uint32_t word[2] = {wnext[0], wnext[1]};
      if (s + 1 < nstages) load_words(s + 1);
      if (dead) continue;
      if (!mbar_wait_ns(&full[st], (gs / STAGES) & 1, wait_ns)) {
        dead = true;
        if (lane == 0) set_status(status, PIE_STATUS_TIMEOUT);
        continue;
      }
      const int unit = warp * kWarpSlots;  // this warp's first row within the stage
      const int unit_base = kb + s * kStageSlots + unit;
      const int nvalid = min(kWarpSlots, ke - unit_base);
      if (nvalid > 0) {
        const uint32_t kbase = ring_s + st * STAGE_BYTES;
        const uint32_t vbase = kbase + 2 * HALF_BYTES;
        if (nvalid < kWarpSlots) {
          // V rows past the visible end hold whatever the stage held before:
          // zero them so that their zero probabilities stay zero in P V
          uint8_t* vrow = ring + st * STAGE_BYTES + 2 * HALF_BYTES;
          for (int i = lane; i < (kWarpSlots - nvalid) * 16; i += 32) {
            const int rr = unit + nvalid + (i >> 4), h = (i >> 3) & 1, ch = i & 7;
            *reinterpret_cast<uint4*>(vrow + h * HALF_BYTES + rr * 128 + ch * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();  // the stage is later rewritten by the copy engine
          __syncwarp();
        }
        // ---- S^T = K Q^T; A matrices: (slots 0-7, d chunk 2k), (8-15, 2k),
        // (0-7, 2k+1), (8-15, 2k+1)
        float cc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          // Q^T fragments of steps 2kk and 2kk + 1: matrices (queries 0-7, chunk 4kk + mi)
          uint32_t b[4];
          const int qc = 4 * kk + mi;
          ldsm_x4(qs_s + mr * 256 + ((qc ^ mr) << 4), b[0], b[1], b[2], b[3]);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int k = 2 * kk + h;
            uint32_t a0, a1, a2, a3;
            ldsm_x4(dm::chunk_addr(kbase, unit + (mi & 1) * 8 + mr, 2 * k + (mi >> 1)), a0, a1, a2,
                    a3);
            dm::mma16816(cc, a0, a1, a2, a3, b[2 * h], b[2 * h + 1]);
          }
        }
        // cc[e]: slot g + 8 (e >> 1) of the unit, query 2t + (e & 1)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int cs = g + 8 * (e >> 1), i = e & 1;
          const bool vis = valid_q[i] && cs < nvalid &&
                           (mrow[i] ? ((word[i] >> cs) & 1u) != 0 : unit_base + cs <= slot_lim[i]);
          cc[e] = vis ? cc[e] : -INFINITY;
        }
        float mt[2] = {fmaxf(cc[0], cc[2]), fmaxf(cc[1], cc[3])};
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mt[0] = fmaxf(mt[0], __shfl_xor_sync(0xffffffffu, mt[0], off));
          mt[1] = fmaxf(mt[1], __shfl_xor_sync(0xffffffffu, mt[1], off));
        }
        float m_new[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float mti = mt[i] * scale_log2;  // scale > 0: the maximum commutes with it
          m_new[i] = m_used[i];
          if (m_used[i] == -INFINITY || mti > m_used[i] + 8.f) m_new[i] = fmaxf(m_used[i], mti);
        }
        if (__any_sync(0xffffffffu, m_new[0] != m_used[0] || m_new[1] != m_used[1])) {
          float alpha[2];
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            alpha[i] = (m_new[i] == m_used[i]) ? 1.f : ex2(m_used[i] - m_new[i]);
            l_part[i] *= alpha[i];
            m_used[i] = m_new[i];
          }
#pragma unroll
          for (int n = 0; n < 8; ++n) {
            o[n][0] *= alpha[0];
            o[n][1] *= alpha[1];
            o[n][2] *= alpha[0];
            o[n][3] *= alpha[1];
          }
        }
        const float neg_m[2] = {m_used[0] == -INFINITY ? 0.f : -m_used[0],
                                m_used[1] == -INFINITY ? 0.f : -m_used[1]};
        float p[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) p[e] = ex2(fmaf(cc[e], scale_log2, neg_m[e & 1]));
        l_part[0] += p[0] + p[2];
        l_part[1] += p[1] + p[3];
        // P^T rows (slots) g and g + 8 as two 8 x 8 bf16 matrices, transposed
        // in registers into the B fragments of P^T: b0 = P[g][2t, 2t+1],
        // b1 = P[g][8 + 2t, 9 + 2t]
        const uint32_t pb0 = dm::movmatrix_t(dm::pack_bf16(p[0], p[1]));
        const uint32_t pb1 = dm::movmatrix_t(dm::pack_bf16(p[2], p[3]));
        // ---- O^T += V^T P^T; A matrices (ldmatrix.trans of V rows): (slots
        // 0-7, d chunk 2n), (0-7, 2n+1), (8-15, 2n), (8-15, 2n+1)
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4_t(dm::chunk_addr(vbase, unit + (mi >> 1) * 8 + mr, 2 * n + (mi & 1)), a0, a1,
                    a2, a3);
          dm::mma16816(o[n], a0, a1, a2, a3, pb0, pb1);
        }
      }
      // the item's last stage stays held: its buffer is the merge's scratch
      if (s + 1 < nstages) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }
    }

    // ---- merge the 4 warps' states into the item's partials, through the
    // held last stage (an item with no stage has only empty states)
    float l_q[2] = {l_part[0], l_part[1]};
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l_q[0] += __shfl_xor_sync(0xffffffffu, l_q[0], off);
      l_q[1] += __shfl_xor_sync(0xffffffffu, l_q[1], off);
    }
    if (nstages == 0) {
      for (int i = threadIdx.x; i < NQ * D; i += WARPS * 32) {
        m.part_o[int64_t(it.part_base + i / D) * D + i % D] = 0.f;
        if (i % D == 0) m.part_ml[it.part_base + i / D] = make_float2(-INFINITY, 0.f);
      }
      continue;
    }
    const int held = (gs - 1) % STAGES;
    float* mw = reinterpret_cast<float*>(ring + held * STAGE_BYTES);  // [WARPS][NQ]
    float* lw = mw + WARPS * NQ;                                      // [WARPS][NQ]
    float* ow = lw + WARPS * NQ;                                      // [WARPS][NQ][D]
    asm volatile("bar.sync 1, %0;" ::"n"(WARPS * 32) : "memory");  // every warp's reads of the stage
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int q = 2 * t + i;
      if (q < NQ) {
        if (g == 0) {
          mw[warp * NQ + q] = m_used[i];
          lw[warp * NQ + q] = l_q[i];
        }
        float* orow = ow + (warp * NQ + q) * D;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          orow[16 * n + g] = o[n][i];
          orow[16 * n + g + 8] = o[n][2 + i];
        }
      }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(WARPS * 32) : "memory");
    for (int i = threadIdx.x; i < NQ * D; i += WARPS * 32) {
      const int qq = i / D, cc = i % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < WARPS; ++w) M = fmaxf(M, mw[w * NQ + qq]);
      float O = 0.f, Ls = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < WARPS; ++w) {
          const float mwv = mw[w * NQ + qq];
          const float f = mwv == -INFINITY ? 0.f : ex2(mwv - M);
          O = fmaf(f, ow[(w * NQ + qq) * D + cc], O);
          Ls = fmaf(f, lw[w * NQ + qq], Ls);
        }
      }
      m.part_o[int64_t(it.part_base + qq) * D + cc] = O;
      if (cc == 0) m.part_ml[it.part_base + qq] = make_float2(M, Ls);
    }
    // the held stage back to the producer once every warp has read its merge
    // data (generic writes into a buffer the copy engine rewrites next)
    fence_proxy_async_smem();
    asm volatile("bar.sync 1, %0;" ::"n"(WARPS * 32) : "memory");
    if (lane == 0 && !dead) mbar_arrive(&empty[held]);
  }
}

template <int NQ>
static cudaError_t launch_nq(const pie_fwd_plan_t& p, const void* q_rot,
                             const uint32_t* mask_words, uint32_t* status, const CUtensorMap& km,
                             const CUtensorMap& vm, const CUtensorMap& kgm, const CUtensorMap& vgm,
                             cudaStream_t s) {
  static std::atomic<uint64_t> configured{0};  // per instantiation and device
  cudaError_t e = set_smem_limit(attend_decode_mma_kernel<NQ>, dm::SMEM, configured);
  if (e != cudaSuccess) return e;
  DevMeta m = p.dev;
  test_wait_hook(&m.test_stall, &m.test_wait_us);
  // a plan's work counter: a persistent grid of three CTAs per SM; without
  // one (the no-allocation decode, the decode loop), fixed runs of items
  const int per = p.dec_items_per_cta > 0 ? p.dec_items_per_cta : 1;
  const int grid = p.dev.dec_work ? std::min(p.num_dec_items, 3 * std::max(1, p.dev.num_sms))
                                  : (p.num_dec_items + per - 1) / per;
  return launch_dependent(attend_decode_mma_kernel<NQ>, dim3(grid), dim3(dm::THREADS),
                          dm::SMEM, s, true, m, p.desc.num_q_heads, p.desc.num_kv_heads, p.G,
                          p.desc.page_size, p.desc.sm_scale * dm::kLog2e,
                          static_cast<const __nv_bfloat16*>(q_rot), mask_words,
                          tc_kv_tile(p.tc_nt), p.num_dec_items, per, status, km, vm, kgm, vgm);
}

// bf16 pools with head_dim 128 whose rows (pool pages x kv heads x page
// size) fit the tensor copies' 32-bit row coordinate
bool decode_mma_supported(const pie_fwd_plan_t& p) {
  const int64_t rows =
      static_cast<int64_t>(p.dev.num_pool_pages) * p.desc.num_kv_heads * p.desc.page_size;
  return p.desc.dtype == PIE_BF16 && p.desc.head_dim == dm::D && p.nq <= 8 && rows > 0 &&
         rows <= INT32_MAX;
}

cudaError_t launch_attend_decode_mma(const pie_fwd_plan_t& p, const void* q_rot,
                                     const void* k_pool, const void* v_pool,
                                     const uint32_t* mask_words, uint32_t* status,
                                     cudaStream_t s) {
  const int Hkv = p.desc.num_kv_heads, P = p.desc.page_size;
  CUtensorMap km, vm;
  const cuuint64_t dims[2] = {cuuint64_t(dm::D), cuuint64_t(p.dev.num_pool_pages) * Hkv * P};
  const cuuint64_t str[1] = {cuuint64_t(dm::D) * 2};
  const cuuint32_t box[2] = {64, cuuint32_t(P)};
  if (!tc::make_map(&km, k_pool, 2, dims, str, box)) return cudaErrorInvalidValue;
  if (!tc::make_map(&vm, v_pool, 2, dims, str, box)) return cudaErrorInvalidValue;
  // one-row boxes for the gathers of scattered lists
  CUtensorMap kgm = km, vgm = vm;
  if (p.dec_lists) {
    const cuuint32_t box1[2] = {64, 1};
    if (!tc::make_map(&kgm, k_pool, 2, dims, str, box1)) return cudaErrorInvalidValue;
    if (!tc::make_map(&vgm, v_pool, 2, dims, str, box1)) return cudaErrorInvalidValue;
  }
  switch (p.nq) {
    case 2: return launch_nq<2>(p, q_rot, mask_words, status, km, vm, kgm, vgm, s);
    case 4: return launch_nq<4>(p, q_rot, mask_words, status, km, vm, kgm, vgm, s);
    default: return launch_nq<8>(p, q_rot, mask_words, status, km, vm, kgm, vgm, s);
  }
}

}  // namespace pie
