// Step 2-3 of a ForwardPass for lanes with few query vectors per kv head
// (decode rows, short drafts): split-KV grouped-query attention over paged
// K/V (Pie "The forward pass": State geometry kv_len; Attention masks).
//
// Decode attention is bound by HBM: every visible slot's K and V head rows
// are read once and used by the NQ query vectors of the GQA group.  The
// kernel therefore
//   * streams pages through a ring of shared-memory stages with 1-D TMA bulk
//     copies (one copy per (page, kv head) block, contiguous in the
//     [page][kv head][slot][d] pools), completed on mbarriers, issued by a
//     dedicated producer warp with an evict-first L2 hint;
//   * lets each of 4 compute warps own 16 slots of every 64-slot stage, with
//     its own online-softmax state, so the main loop needs no CTA barrier;
//   * keeps the NQ query vectors in registers split along d (16 bytes per
//     lane) and reduces the NQ x 16 partial dot products of a warp with a
//     transposed butterfly (each round halves the values a lane holds), so
//     that scoring a slot costs about two shuffles instead of log2(lanes)
//     per query;
//   * accumulates P.V with lanes split along d and probabilities broadcast
//     from a per-warp shared buffer.
// Scores are kept in the log2 domain (q pre-scaled by sm_scale * log2 e).
// Each work item writes one partial (max, sum, unnormalised output) per
// query vector; the combine kernel (combine.cu) merges an item's chunks.

#include "common.cuh"

namespace pie {

constexpr float kLog2e = 1.4426950408889634f;

template <typename T, int D, int NQ>
struct DecCfg {
  static constexpr int EPL = 16 / sizeof(T);      // q/K elements per lane (one 16-byte vector)
  static constexpr int LPR = D / EPL;             // lanes covering one K row
  static constexpr int RPS = 32 / LPR;            // K rows per warp step
  static constexpr int STEPS = kWarpSlots / RPS;  // steps per 16-slot unit
  static constexpr int NV = STEPS * NQ;           // partial dot products per lane
  static constexpr int E = NV / LPR;              // scores per lane after the reduction
  static constexpr int DPL = D / 32;              // output elements per lane in P.V
  static constexpr int WARPS = 4;                 // compute warps (+1 producer warp)
  static constexpr int THREADS = (WARPS + 1) * 32;
  static constexpr int ROW_BYTES = D * sizeof(T);
  static constexpr int STAGE_BYTES = 2 * kStageSlots * ROW_BYTES;  // K + V
  // a 64 KB ring (2 to 4 stages): HBM latency needs far less in flight per
  // SM than three CTAs' rings, and three resident CTAs (15 warps) hide the
  // compute warps' latencies better than deeper rings
  static constexpr int STAGES = (65536 / STAGE_BYTES) < 2 ? 2
                                : (65536 / STAGE_BYTES) > 4 ? 4 : (65536 / STAGE_BYTES);
  static constexpr int PBUF_FLOATS = WARPS * kWarpSlots * NQ;
  static constexpr int ABUF_FLOATS = WARPS * NQ;
  static constexpr size_t SMEM = size_t(STAGES) * STAGE_BYTES +
                                 sizeof(float) * (PBUF_FLOATS + ABUF_FLOATS) +
                                 sizeof(uint64_t) * 2 * STAGES;
  // resident CTAs per SM the registers are capped for (NQ = 8 keeps its
  // registers; shared memory decides the rest)
  static constexpr int MIN_BLOCKS = NQ >= 8 ? 1 : (SMEM <= 70000 ? 3 : (SMEM <= 110000 ? 2 : 1));
  static_assert(E == NQ / 2, "reduction layout assumes E = NQ / 2");
  static_assert(kWarpSlots % RPS == 0, "unit must hold whole steps");
  static_assert(size_t(WARPS) * NQ * (D + 2) * 4 <= size_t(STAGES) * STAGE_BYTES,
                "merge buffers must fit in the stage ring");
};

// Transposed butterfly: v[0..N) partial sums per lane; after log2(LPR)
// rounds lane j of its row group holds the complete sums of entries
// [j * N/LPR, (j+1) * N/LPR) in v[0 .. N/LPR).
template <int N, int OFF>
struct TReduce {
  static __device__ __forceinline__ void run(float* v, int j) {
    const bool upper = (j & OFF) != 0;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      const float send = upper ? v[i] : v[i + N / 2];
      const float keep = upper ? v[i + N / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
    }
    TReduce<N / 2, OFF / 2>::run(v, j);
  }
};
template <int N>
struct TReduce<N, 0> {
  static __device__ __forceinline__ void run(float*, int) {}
};

__device__ __forceinline__ float warp_max_pairs(float x) {
#pragma unroll
  for (int off = 2; off < 32; off <<= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
  return x;
}
__device__ __forceinline__ float warp_sum_pairs(float x) {
#pragma unroll
  for (int off = 2; off < 32; off <<= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// Load DPL consecutive elements (4, 8 or 16 bytes) as floats.
template <typename T, int DPL>
__device__ __forceinline__ void load_dpl(const T* p, float* f) {
  if constexpr (sizeof(T) * DPL == 16) {
    unpack16<T>(*reinterpret_cast<const uint4*>(p), f);
  } else if constexpr (sizeof(T) * DPL == 8) {
    unpack8<T>(*reinterpret_cast<const uint2*>(p), f);
  } else {
    static_assert(sizeof(T) * DPL == 4, "unsupported lane width");
    const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
    if constexpr (sizeof(T) == 2) {
      f[0] = __uint_as_float(u << 16);
      f[1] = __uint_as_float(u & 0xFFFF0000u);
    } else {
      f[0] = __uint_as_float(u);
    }
  }
}

// NQ probabilities of one slot from the per-warp buffer (16-byte aligned for
// NQ >= 4, 8-byte for NQ = 2) as vector loads.
template <int NQ>
__device__ __forceinline__ void load_probs(const float* p, float* f) {
  if constexpr (NQ == 2) {
    const float2 v = *reinterpret_cast<const float2*>(p);
    f[0] = v.x;
    f[1] = v.y;
  } else {
#pragma unroll
    for (int i = 0; i < NQ; i += 4) {
      const float4 v = *reinterpret_cast<const float4*>(p + i);
      f[i] = v.x;
      f[i + 1] = v.y;
      f[i + 2] = v.z;
      f[i + 3] = v.w;
    }
  }
}

template <typename T, int D, int NQ>
__global__ void __launch_bounds__(DecCfg<T, D, NQ>::THREADS, DecCfg<T, D, NQ>::MIN_BLOCKS)
    attend_decode_kernel(
    DevMeta m, int Hq, int Hkv, int G, int P, float scale_log2, const T* q_rot,
    const T* k_pool, const T* v_pool, const uint32_t* mask_words, uint32_t* status) {
  using C = DecCfg<T, D, NQ>;
  extern __shared__ __align__(128) uint8_t smem[];
  T* ring = reinterpret_cast<T*>(smem);
  float* pbuf = reinterpret_cast<float*>(smem + size_t(C::STAGES) * C::STAGE_BYTES);
  float* abuf = pbuf + C::PBUF_FLOATS;
  uint64_t* full = reinterpret_cast<uint64_t*>(abuf + C::ABUF_FLOATS);
  uint64_t* empty = full + C::STAGES;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::WARPS);
    }
    fence_barrier_init();
  }
  __syncthreads();
  // The barrier set-up above overlaps the kernel before; everything below,
  // the work item included, is read after the wait: the items may come from
  // a kernel queued just before this one (the decode loop's geometry step,
  // the no-allocation entry point's item kernel), whose writes are only
  // guaranteed visible once griddepcontrol.wait has returned.
  grid_dep_wait();
  grid_dep_launch();
  const DecItem it = m.dec_items[blockIdx.x];
  const int kb = it.kv_begin, ke = it.kv_end;
  const int nstages = ke > kb ? (ke - kb + kStageSlots - 1) / kStageSlots : 0;
  const int nqv = it.nrows * G;  // valid query vectors

  // every wait gives up after the limit (the test hook may shorten it)
  const uint64_t wait_ns = m.test_wait_us ? uint64_t(m.test_wait_us) * 1000ull : kWaitLimitNs;

  if (warp == C::WARPS) {
    // ---------------- producer warp: TMA bulk copies of K/V pages ----------
    // Lanes 2i and 2i + 1 copy the K and the V block of page (stage start /
    // P + i) of every stage (a warp's copies issue one after another, so
    // each comes from its own lane); the page ids of the next stage are
    // fetched while this one is issued, so no copy waits on a dependent
    // global load.  A page id outside the pool is not copied (its slots keep
    // whatever the stage held) and sets PIE_STATUS_BOUNDS: page tables that
    // device code supplies are checked here.
    const uint64_t pol = policy_evict_first();
    const int32_t* pages = m.page_ids + m.page_indptr[it.lane];
    const int64_t head_stride = int64_t(P) * D;  // elements per (page, kv head) block
    const uint32_t blk = uint32_t(P) * C::ROW_BYTES;
    auto page_of = [&](int s) -> int64_t {
      const int sb = kb + s * kStageSlots;
      const int p0 = sb / P, p1 = (min(sb + kStageSlots, ke) - 1) / P;
      return (lane >> 1) <= p1 - p0 ? int64_t(pages[p0 + (lane >> 1)]) : 0;
    };
    int64_t pid = nstages > 0 ? page_of(0) : 0;
    for (int s = 0; s < nstages; ++s) {
      // test hook: stop before this stage (no copy of it is ever issued, so
      // none is in flight when the compute warps' waits for it expire)
      if (s == m.test_stall - 1) break;
      const int st = s % C::STAGES, use = s / C::STAGES;
      if (use > 0 && !mbar_wait_ns(&empty[st], (use - 1) & 1, wait_ns)) {
        if (lane == 0) set_status(status, PIE_STATUS_TIMEOUT);
        break;
      }
      const int sb = kb + s * kStageSlots;
      const int se = min(sb + kStageSlots, ke);
      const int p0 = sb / P, p1 = (se - 1) / P;
      const bool mine = (lane >> 1) <= p1 - p0;
      const bool in_pool = pid >= 0 && pid < m.num_pool_pages;
      const bool issue = mine && in_pool;
      const uint32_t copies = __popc(__ballot_sync(0xffffffffu, issue));
      if (lane == 0) {
        if (copies != 2u * uint32_t(p1 - p0 + 1)) set_status(status, PIE_STATUS_BOUNDS);
        mbar_arrive_expect_tx(&full[st], blk * copies);
      }
      __syncwarp();
      if (issue) {
        const bool is_v = lane & 1;
        T* dst = ring + size_t(st) * 2 * kStageSlots * D + (is_v ? kStageSlots * D : 0);
        const int64_t src = (pid * Hkv + it.kv_head) * head_stride;
        const int off = ((p0 + (lane >> 1)) * P - sb) * D;
        bulk_g2s_hint(dst + off, (is_v ? v_pool : k_pool) + src, blk, &full[st], pol);
      }
      if (s + 1 < nstages) pid = page_of(s + 1);
    }
    return;
  }

  // ---------------- compute warps ---------------------------------------------
  const int j = lane % C::LPR;   // lane within its K row group
  const int rg = lane / C::LPR;  // row group (slot within a step)

  float qr[NQ][C::EPL];
#pragma unroll
  for (int qq = 0; qq < NQ; ++qq) {
    const int qv = min(qq, nqv - 1);
    const int row = it.row0 + qv / G, head = it.kv_head * G + qv % G;
    const uint4 u =
        *reinterpret_cast<const uint4*>(q_rot + (int64_t(row) * Hq + head) * D + j * C::EPL);
    unpack16<T>(u, qr[qq]);
#pragma unroll
    for (int e = 0; e < C::EPL; ++e) qr[qq][e] *= scale_log2;
  }
  // the E query vectors whose scores this lane holds after the reduction
  bool qvalid[C::E];
  int slot_lim[C::E];
  int64_t mbase[C::E];
#pragma unroll
  for (int e = 0; e < C::E; ++e) {
    const int qq = (j & 1) * C::E + e;
    qvalid[e] = qq < nqv;
    const int row = it.row0 + min(qq, nqv - 1) / G;
    slot_lim[e] = m.slots[row];
    mbase[e] = mask_words ? m.mask_word_indptr[row] : 0;
  }

  float m_run[C::E], l_run[C::E];
#pragma unroll
  for (int e = 0; e < C::E; ++e) {
    m_run[e] = -INFINITY;
    l_run[e] = 0.f;
  }
  float acc[NQ][C::DPL];
#pragma unroll
  for (int qq = 0; qq < NQ; ++qq)
#pragma unroll
    for (int c = 0; c < C::DPL; ++c) acc[qq][c] = 0.f;

  float* my_p = pbuf + warp * kWarpSlots * NQ;
  float* my_a = abuf + warp * NQ;
  const int s_in_unit = (j >> 1) * C::RPS + rg;
  bool timed_out = false;

  for (int s = 0; s < nstages; ++s) {
    const int st = s % C::STAGES;
    if (!mbar_wait_ns(&full[st], (s / C::STAGES) & 1, wait_ns)) {
      timed_out = true;
      break;
    }
    const int unit_base = kb + s * kStageSlots + warp * kWarpSlots;
    const int nvalid = min(kWarpSlots, ke - unit_base);
    if (nvalid > 0) {
      const T* Ks = ring + size_t(st) * 2 * kStageSlots * D + warp * kWarpSlots * D;
      const T* Vs = Ks + kStageSlots * D;
      // ---- scores: NQ x 16 dot products, reduced across the row group
      float part[C::NV];
#pragma unroll
      for (int t = 0; t < C::STEPS; ++t) {
        float kf[C::EPL];
        unpack16<T>(*reinterpret_cast<const uint4*>(Ks + (t * C::RPS + rg) * D + j * C::EPL), kf);
        // pairs of d per packed FMA, the two halves added at the end
#pragma unroll
        for (int qq = 0; qq < NQ; ++qq) {
          float a0 = 0.f, a1 = 0.f;
#pragma unroll
          for (int e = 0; e < C::EPL; e += 2)
            ffma2(a0, a1, qr[qq][e], qr[qq][e + 1], kf[e], kf[e + 1], a0, a1);
          part[t * NQ + qq] = a0 + a1;
        }
      }
      TReduce<C::NV, C::LPR / 2>::run(part, j);
      // ---- online softmax for this warp's 16 slots
      const int s_abs = unit_base + s_in_unit;
      uint32_t word[C::E];
#pragma unroll
      for (int e = 0; e < C::E; ++e)
        word[e] = (mask_words && s_in_unit < nvalid) ? mask_words[mbase[e] + (s_abs >> 5)] : 0u;
#pragma unroll
      for (int e = 0; e < C::E; ++e) {
        const bool in = qvalid[e] && s_in_unit < nvalid;
        const bool vis = in && (mask_words ? ((word[e] >> (s_abs & 31)) & 1u) != 0
                                           : s_abs <= slot_lim[e]);
        const float sc = vis ? part[e] : -INFINITY;
        const float m_new = fmaxf(m_run[e], warp_max_pairs(sc));
        const bool none = m_new == -INFINITY;
        const float alpha = none ? 1.f : ex2(m_run[e] - m_new);
        const float p = vis ? ex2(sc - m_new) : 0.f;
        l_run[e] = l_run[e] * alpha + warp_sum_pairs(p);
        m_run[e] = m_new;
        const int qq = (j & 1) * C::E + e;
        my_p[s_in_unit * NQ + qq] = p;
        if (lane < 2) my_a[qq] = alpha;
      }
      __syncwarp();
      // ---- P.V with lanes split along d
#pragma unroll
      for (int qq = 0; qq < NQ; ++qq) {
        const float a = my_a[qq];
#pragma unroll
        for (int c = 0; c < C::DPL; ++c) acc[qq][c] *= a;
      }
      for (int sl = 0; sl < nvalid; ++sl) {
        float vf[C::DPL];
        load_dpl<T, C::DPL>(Vs + sl * D + lane * C::DPL, vf);
        float pq[NQ];
        load_probs<NQ>(my_p + sl * NQ, pq);
        // pairs of output elements per packed FMA
#pragma unroll
        for (int qq = 0; qq < NQ; ++qq)
#pragma unroll
          for (int c = 0; c < C::DPL; c += 2)
            ffma2(acc[qq][c], acc[qq][c + 1], pq[qq], pq[qq], vf[c], vf[c + 1], acc[qq][c],
                  acc[qq][c + 1]);
      }
      __syncwarp();
    }
    if (lane == 0) mbar_arrive(&empty[st]);
  }
  if (timed_out && lane == 0) set_status(status, PIE_STATUS_TIMEOUT);

  // ---- merge the 4 warps' states (ring memory is free: every stage was
  // consumed, so no copy is in flight) and write the item's partials
  asm volatile("bar.sync 1, %0;" ::"n"(C::WARPS * 32) : "memory");
  float* mw = reinterpret_cast<float*>(smem);   // [WARPS][NQ]
  float* lw = mw + C::WARPS * NQ;               // [WARPS][NQ]
  float* ow = lw + C::WARPS * NQ;               // [WARPS][NQ][D]
  if (rg == 0 && j < 2) {
#pragma unroll
    for (int e = 0; e < C::E; ++e) {
      mw[warp * NQ + j * C::E + e] = m_run[e];
      lw[warp * NQ + j * C::E + e] = l_run[e];
    }
  }
#pragma unroll
  for (int qq = 0; qq < NQ; ++qq)
#pragma unroll
    for (int c = 0; c < C::DPL; ++c) ow[(warp * NQ + qq) * D + lane * C::DPL + c] = acc[qq][c];
  asm volatile("bar.sync 1, %0;" ::"n"(C::WARPS * 32) : "memory");
  for (int idx = threadIdx.x; idx < NQ * D; idx += C::WARPS * 32) {
    const int qq = idx / D, c = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < C::WARPS; ++w) M = fmaxf(M, mw[w * NQ + qq]);
    float O = 0.f, Ls = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < C::WARPS; ++w) {
        const float f = ex2(mw[w * NQ + qq] - M);
        O = fmaf(f, ow[(w * NQ + qq) * D + c], O);
        Ls = fmaf(f, lw[w * NQ + qq], Ls);
      }
    }
    m.part_o[int64_t(it.part_base + qq) * D + c] = O;
    if (c == 0) m.part_ml[it.part_base + qq] = make_float2(M, Ls);
  }
}

template <typename T, int D, int NQ>
static cudaError_t launch_dec(const pie_fwd_plan_t& p, const void* q_rot, const void* k_pool,
                              const void* v_pool, const uint32_t* mask_words, uint32_t* status,
                              cudaStream_t s) {
  using C = DecCfg<T, D, NQ>;
  static std::atomic<uint64_t> configured{0};  // per instantiation and device
  cudaError_t e = set_smem_limit(attend_decode_kernel<T, D, NQ>, int(C::SMEM), configured);
  if (e != cudaSuccess) return e;
  DevMeta m = p.dev;
  test_wait_hook(&m.test_stall, &m.test_wait_us);
  return launch_dependent(attend_decode_kernel<T, D, NQ>, dim3(p.num_dec_items), dim3(C::THREADS),
                          C::SMEM, s, true, m, p.desc.num_q_heads, p.desc.num_kv_heads, p.G,
                          p.desc.page_size, p.desc.sm_scale * kLog2e, static_cast<const T*>(q_rot),
                          static_cast<const T*>(k_pool), static_cast<const T*>(v_pool), mask_words,
                          status);
}

template <typename T, int D>
static cudaError_t launch_dec_nq(const pie_fwd_plan_t& p, const void* q_rot, const void* k_pool,
                                 const void* v_pool, const uint32_t* mask_words, uint32_t* status,
                                 cudaStream_t s) {
  switch (p.nq) {
    case 2: return launch_dec<T, D, 2>(p, q_rot, k_pool, v_pool, mask_words, status, s);
    case 4: return launch_dec<T, D, 4>(p, q_rot, k_pool, v_pool, mask_words, status, s);
    default: return launch_dec<T, D, 8>(p, q_rot, k_pool, v_pool, mask_words, status, s);
  }
}

cudaError_t launch_attend_decode(const pie_fwd_plan_t& p, const void* q_rot, const void* k_pool,
                                 const void* v_pool, const uint32_t* mask_words,
                                 uint32_t* status, cudaStream_t s) {
  if (decode_mma_supported(p))
    return launch_attend_decode_mma(p, q_rot, k_pool, v_pool, mask_words, status, s);
  // items that walk compacted lists are only planned for passes the kernel
  // above takes
  if (p.dec_lists) return cudaErrorNotSupported;
  const bool bf = p.desc.dtype == PIE_BF16;
  if (p.desc.head_dim == 128)
    return bf ? launch_dec_nq<__nv_bfloat16, 128>(p, q_rot, k_pool, v_pool, mask_words, status, s)
              : launch_dec_nq<float, 128>(p, q_rot, k_pool, v_pool, mask_words, status, s);
  return bf ? launch_dec_nq<__nv_bfloat16, 64>(p, q_rot, k_pool, v_pool, mask_words, status, s)
            : launch_dec_nq<float, 64>(p, q_rot, k_pool, v_pool, mask_words, status, s);
}

}  // namespace pie
