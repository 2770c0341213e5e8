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
// here each compute warp takes its 16 slots of a 64-slot stage with
//   * S = Q K^T as 16 x 8 x 16 bf16 MMAs (the query vectors are the rows of
//     A, padded to 16 with zeros; two 8-slot column tiles, eight 16-wide
//     steps over d), K fragments read with ldmatrix;
//   * the online softmax on the accumulator fragments: each row's 16 scores
//     sit in the four lanes of its quad (two shuffles for the maximum), and
//     the running maximum used for the exponent only moves when a tile's
//     maximum exceeds it by more than 2^8, so the output is rarely rescaled;
//   * O += P V as 16 MMAs, P (bf16) taken straight from the score fragments
//     as the A operand, V fragments read with ldmatrix.trans.
// That is about 100 warp instructions per warp and stage where the scalar
// kernel needs about 900.  The fragments need K and V rows in shared memory
// without bank conflicts between slots, so the producer warp copies each
// (page, kv head) block as two 2-D tensor boxes of P rows x 128 bytes (one
// per half of d) with the 128-byte swizzle; with two CTAs per SM, each with
// a three-stage ring, those copies stream at the copy bandwidth.
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
constexpr int STAGES = 3;                          // a 96 KB ring: two CTAs per SM
constexpr int SMEM = STAGES * STAGE_BYTES + 1024 + 2 * STAGES * 8;  // + alignment + barriers
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

// D[g][2t..2t+1] += A[g][.] B[.][2t..2t+1] for a 16 x 8 x 16 bf16 MMA whose
// A rows 8..15 are zero (a1 = a3 = 0): only the accumulators of rows 0..7
// are kept; those of rows 8..15 stay zero and are discarded.
__device__ __forceinline__ void mma_top(float& d0, float& d1, uint32_t a0, uint32_t a2, uint32_t b0,
                                        uint32_t b1) {
  float z0, z1;
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %10, %10};"
      : "+f"(d0), "+f"(d1), "=f"(z0), "=f"(z1)
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1), "f"(0.f));
  (void)z0;
  (void)z1;
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

template <int NQ>
__global__ void __launch_bounds__(dm::THREADS, 2) attend_decode_mma_kernel(
    DevMeta m, int Hq, int Hkv, int G, int P, float scale_log2, const __nv_bfloat16* q_rot,
    const uint32_t* mask_words, uint32_t* status, const __grid_constant__ CUtensorMap kmap,
    const __grid_constant__ CUtensorMap vmap) {
  using namespace dm;
  static_assert(NQ <= 8, "query vectors of an item fill at most the top 8 MMA rows");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], WARPS);
    }
    fence_barrier_init();
  }
  __syncthreads();
  // everything below, the work item included, is read after the wait (the
  // items may come from a kernel queued just before this one)
  grid_dep_wait();
  grid_dep_launch();
  const DecItem it = m.dec_items[blockIdx.x];
  const int kb = it.kv_begin, ke = it.kv_end;
  const int nstages = ke > kb ? (ke - kb + kStageSlots - 1) / kStageSlots : 0;
  const int nqv = it.nrows * G;
  const uint64_t wait_ns = m.test_wait_us ? uint64_t(m.test_wait_us) * 1000ull : kWaitLimitNs;

  if (warp == WARPS) {
    // ---------------- producer warp: 2-D tensor copies of K/V pages -----------
    // Lane 4i + c copies block c (K half 0, K half 1, V half 0, V half 1) of
    // page (stage start / P + i); a stage spans 64 / P pages (at most 8).
    // The page ids of the next stage are fetched while this one is issued.
    // A page id outside the pool is not copied and sets PIE_STATUS_BOUNDS.
    const uint64_t pol = policy_evict_first();
    const int32_t* pages = m.page_ids + m.page_indptr[it.lane];
    const int c = lane & 3, pi = lane >> 2;
    auto page_of = [&](int s) -> int64_t {
      const int sb = kb + s * kStageSlots;
      const int p0 = sb / P, p1 = (min(sb + kStageSlots, ke) - 1) / P;
      return pi <= p1 - p0 ? int64_t(pages[p0 + pi]) : 0;
    };
    int64_t pid = nstages > 0 ? page_of(0) : 0;
    for (int s = 0; s < nstages; ++s) {
      if (s == m.test_stall - 1) break;  // test hook: no copy of this stage is ever issued
      const int st = s % STAGES, use = s / STAGES;
      if (use > 0 && !mbar_wait_ns(&empty[st], (use - 1) & 1, wait_ns)) {
        if (lane == 0) set_status(status, PIE_STATUS_TIMEOUT);
        break;
      }
      const int sb = kb + s * kStageSlots;
      const int se = min(sb + kStageSlots, ke);
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
        uint8_t* dst = ring + st * STAGE_BYTES + (c >> 1) * 2 * HALF_BYTES + (c & 1) * HALF_BYTES +
                       ((p0 + pi) * P - sb) * 128;
        tc::tma_2d(dst, (c >> 1) ? &vmap : &kmap, 64 * (c & 1),
                   int((pid * Hkv + it.kv_head) * P), &full[st], pol);
      }
      if (s + 1 < nstages) pid = page_of(s + 1);
    }
    return;
  }

  // ---------------- compute warps ---------------------------------------------
  const int g = lane >> 2, t = lane & 3;  // fragment row (query vector) and column pair
  const bool valid_q = g < nqv;
  const int qv = valid_q ? g : 0;
  const int row = it.row0 + qv / G, head = it.kv_head * G + qv % G;
  const int slot_lim = valid_q ? m.slots[row] : -1;
  const uint32_t* mrow = (mask_words && valid_q) ? mask_words + m.mask_word_indptr[row] : nullptr;
  // A fragments of Q (rows 0..7; rows 8..15 are zero): a0 = Q[g][16k + 2t, +1],
  // a2 = Q[g][16k + 2t + 8, +9]
  uint32_t qa[8][2];
  {
    const uint32_t* qp =
        reinterpret_cast<const uint32_t*>(q_rot + (int64_t(row) * Hq + head) * D) + t;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      qa[k][0] = valid_q ? qp[8 * k] : 0u;
      qa[k][1] = valid_q ? qp[8 * k + 4] : 0u;
    }
  }
  float o[16][2];  // O[g][8 n + 2t, +1]
#pragma unroll
  for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = 0.f;
  float m_used = -INFINITY, l_part = 0.f;  // l_part: this lane's share of the row sum
  const uint32_t ring_s = smem_u32(ring);
  // ldmatrix row addresses: lane i serves row i & 7 of matrix i >> 3
  const int mi = lane >> 3, mr = lane & 7;
  bool timed_out = false;

  for (int s = 0; s < nstages; ++s) {
    const int st = s % STAGES;
    if (!mbar_wait_ns(&full[st], (s / STAGES) & 1, wait_ns)) {
      timed_out = true;
      break;
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
          const int r = unit + nvalid + (i >> 4), h = (i >> 3) & 1, ch = i & 7;
          *reinterpret_cast<uint4*>(vrow + h * HALF_BYTES + r * 128 + ch * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();  // the stage is later rewritten by the copy engine
        __syncwarp();
      }
      // ---- S = Q K^T: column tiles of 8 slots (n = 0, 1); scores of row g at
      // unit slots 2t, 2t + 1 (x[0], x[1]) and 8 + 2t, 9 + 2t (x[2], x[3])
      float x[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        // matrices: (slots 0-7, d chunk 2k), (0-7, 2k+1), (8-15, 2k), (8-15, 2k+1)
        uint32_t b0, b1, b2, b3;
        ldsm_x4(dm::chunk_addr(kbase, unit + (mi >> 1) * 8 + mr, 2 * k + (mi & 1)), b0, b1, b2, b3);
        mma_top(x[0], x[1], qa[k][0], qa[k][1], b0, b1);
        mma_top(x[2], x[3], qa[k][0], qa[k][1], b2, b3);
      }
      const uint32_t word = mrow ? (mrow[unit_base >> 5] >> (unit_base & 31)) : ~0u;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int cs = (e >> 1) * 8 + 2 * t + (e & 1);  // slot within the unit
        const bool vis = valid_q && cs < nvalid &&
                         (mrow ? ((word >> cs) & 1u) != 0 : unit_base + cs <= slot_lim);
        x[e] = vis ? x[e] : -INFINITY;
      }
      float mt = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
      mt *= scale_log2;  // scale > 0: the maximum commutes with it
      float m_new = m_used;
      if (m_used == -INFINITY || mt > m_used + 8.f) m_new = fmaxf(m_used, mt);
      if (__any_sync(0xffffffffu, m_new != m_used)) {
        const float alpha = (m_new == m_used) ? 1.f : ex2(m_used - m_new);
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          o[n][0] *= alpha;
          o[n][1] *= alpha;
        }
        l_part *= alpha;
        m_used = m_new;
      }
      const float neg_m = (m_used == -INFINITY) ? 0.f : -m_used;
      float p[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) p[e] = ex2(fmaf(x[e], scale_log2, neg_m));
      l_part += (p[0] + p[1]) + (p[2] + p[3]);
      // P as the A operand of P V: a0 = P[g][2t, +1], a2 = P[g][8 + 2t, +1]
      const uint32_t pa0 = dm::pack_bf16(p[0], p[1]), pa2 = dm::pack_bf16(p[2], p[3]);
      // ---- O += P V: output column tiles n = 2j, 2j + 1 (8 d each)
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        // matrices: (slots 0-7, d chunk 2j), (8-15, 2j), (0-7, 2j+1), (8-15, 2j+1)
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(dm::chunk_addr(vbase, unit + (mi & 1) * 8 + mr, 2 * jj + (mi >> 1)), b0, b1, b2,
                  b3);
        mma_top(o[2 * jj][0], o[2 * jj][1], pa0, pa2, b0, b1);
        mma_top(o[2 * jj + 1][0], o[2 * jj + 1][1], pa0, pa2, b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }
  if (timed_out && lane == 0) set_status(status, PIE_STATUS_TIMEOUT);

  // ---- merge the 4 warps' states (the ring is free: every stage issued was
  // consumed, so no copy is in flight) and write the item's partials
  float l_row = l_part;
  l_row += __shfl_xor_sync(0xffffffffu, l_row, 1);
  l_row += __shfl_xor_sync(0xffffffffu, l_row, 2);
  asm volatile("bar.sync 1, %0;" ::"n"(WARPS * 32) : "memory");
  float* mw = reinterpret_cast<float*>(ring);  // [WARPS][NQ]
  float* lw = mw + WARPS * NQ;                 // [WARPS][NQ]
  float* ow = lw + WARPS * NQ;                 // [WARPS][NQ][D]
  if (g < NQ) {
    if (t == 0) {
      mw[warp * NQ + g] = m_used;
      lw[warp * NQ + g] = l_row;
    }
#pragma unroll
    for (int n = 0; n < 16; ++n)
      *reinterpret_cast<float2*>(ow + (warp * NQ + g) * D + 8 * n + 2 * t) =
          make_float2(o[n][0], o[n][1]);
  }
  asm volatile("bar.sync 1, %0;" ::"n"(WARPS * 32) : "memory");
  for (int idx = threadIdx.x; idx < NQ * D; idx += WARPS * 32) {
    const int qq = idx / D, cc = idx % D;
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
}

template <int NQ>
static cudaError_t launch_nq(const pie_fwd_plan_t& p, const void* q_rot,
                             const uint32_t* mask_words, uint32_t* status, const CUtensorMap& km,
                             const CUtensorMap& vm, cudaStream_t s) {
  static std::atomic<uint64_t> configured{0};  // per instantiation and device
  cudaError_t e = set_smem_limit(attend_decode_mma_kernel<NQ>, dm::SMEM, configured);
  if (e != cudaSuccess) return e;
  DevMeta m = p.dev;
  test_wait_hook(&m.test_stall, &m.test_wait_us);
  return launch_dependent(attend_decode_mma_kernel<NQ>, dim3(p.num_dec_items), dim3(dm::THREADS),
                          dm::SMEM, s, true, m, p.desc.num_q_heads, p.desc.num_kv_heads, p.G,
                          p.desc.page_size, p.desc.sm_scale * dm::kLog2e,
                          static_cast<const __nv_bfloat16*>(q_rot), mask_words, status, km, vm);
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
  switch (p.nq) {
    case 2: return launch_nq<2>(p, q_rot, mask_words, status, km, vm, s);
    case 4: return launch_nq<4>(p, q_rot, mask_words, status, km, vm, s);
    default: return launch_nq<8>(p, q_rot, mask_words, status, km, vm, s);
  }
}

}  // namespace pie
