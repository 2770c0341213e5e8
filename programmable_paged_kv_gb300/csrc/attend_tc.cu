// Step 2-3 of a ForwardPass for lanes with many query vectors per kv head
// (prefill rows, speculative-verify drafts, masked prefill): grouped-query
// attention over paged K/V on the 5th-generation tensor cores (Pie "The
// forward pass": State geometry kv_len; Attention masks).
//
// One CTA handles a work item: up to 128 query vectors (the G heads of a kv
// group for up to 128/G consecutive rows of one lane, head-minor) against
// one chunk of the lane's slots, in 128-slot KV tiles.
//   warp 0  TMA producer: the query tile once (4-D tensor map over q_rot
//           [N][Hkv][G][d]), then per KV tile the K and V blocks of every
//           page in the tile (2-D tensor maps over the pools, one 64-column
//           box per half of d), 128-byte swizzled, double-buffered;
//   warp 1  allocates 512 TMEM columns and issues, from one thread,
//           S = Q K^T (M=128, N=128, K=16 per instruction, operands in shared
//           memory, fp32 accumulator in TMEM; two S buffers so the next
//           tile's scores overlap this tile's softmax) and O += P V (P from
//           shared memory, V used MN-major straight from its tile);
//           tcgen05.commit arrives on mbarriers;
//   warps 2-5  softmax: each thread owns one query row (its TMEM lane),
//           reads 128 scores with one tcgen05.ld, applies the row's
//           visibility (slot-causal or its mask words), keeps the online
//           max/sum in the log2 domain, rescales O in TMEM when the max
//           grows, and writes P (bf16, swizzled) for the P.V product.
// At the end each thread writes its row's partial state (max, sum and the
// unnormalised output) for the combine step.  Every wait is bounded.

#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "tmem128.cuh"

namespace pie {

namespace tc {

constexpr int kThreads = 192;
constexpr int kHalfBytes = 128 * 128;  // 128 rows x 128 bytes: one half of d for a tile
constexpr uint32_t kTmemCols = 512;     // S0 [0,128), S1 [128,256), O [256,384)

struct __align__(1024) Smem {
  uint8_t q[2][kHalfBytes];        // [half of d][query][128 B]
  uint8_t k[2][2][kHalfBytes];     // [stage][half of d][slot][128 B]
  uint8_t v[2][2][kHalfBytes];     // [stage][half of d][slot][128 B]
  uint8_t p[2][kHalfBytes];        // [half of slots][query][128 B]
  uint64_t q_full;
  uint64_t kv_full[2], kv_empty[2];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full, o_done;
  uint32_t tmem_base;
};

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 format: start
// address, leading and stride byte offsets in 16-byte units, descriptor
// version 1, layout type 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t sdesc(const void* p, uint32_t lbo, uint32_t sbo) {
  const uint32_t a = smem_u32(p);
  uint64_t d = uint64_t((a >> 4) & 0x3FFFu);
  d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
  d |= uint64_t((sbo >> 4) & 0x3FFFu) << 32;
  d |= uint64_t(1) << 46;
  d |= uint64_t(2) << 61;
  return d;
}

// Instruction descriptor for kind::f16: bf16 A and B, fp32 accumulator,
// A K-major, B K-major (false) or MN-major (true), N >> 3 and M >> 4.
__host__ __device__ constexpr uint32_t idesc(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id,
                                    uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(id), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float* f) {
  uint32_t r[128];
  asm volatile(PIE_TMEM_LD128_ASM : PIE_TMEM_LD_OUTS : "r"(taddr) : "memory");
#pragma unroll
  for (int i = 0; i < 128; ++i) f[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st128(uint32_t taddr, const float* f) {
  uint32_t r[128];
#pragma unroll
  for (int i = 0; i < 128; ++i) r[i] = __float_as_uint(f[i]);
  asm volatile(PIE_TMEM_ST128_ASM ::"r"(taddr), PIE_TMEM_ST_INS : "memory");
}

__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* map, int x, int y,
                                       uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_4d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                       int w, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
      : "memory");
}

}  // namespace tc

__global__ void __launch_bounds__(tc::kThreads, 1) attend_tc_kernel(
    DevMeta m, int G, int Hkv, int P, float scale_log2, const uint32_t* __restrict__ mask_words,
    uint32_t* status, const __grid_constant__ CUtensorMap qmap,
    const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
  using namespace tc;
  extern __shared__ uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const TcItem it = m.tc_items[blockIdx.x];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kb = it.kv_begin, ke = it.kv_end;
  const int T = ke > kb ? (ke - kb + kTcTileSlots - 1) / kTcTileSlots : 0;
  const int nqv = it.nrows * G;
  constexpr int D = 128;

  if (threadIdx.x == 0) {
    mbar_init(&S.q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.kv_full[i], 1);
      mbar_init(&S.kv_empty[i], 1);
      mbar_init(&S.s_full[i], 1);
      mbar_init(&S.s_free[i], 4);
    }
    mbar_init(&S.p_full, 4);
    mbar_init(&S.o_done, 1);
    fence_barrier_init();
  }
  if (warp == 1 && T > 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&S.tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = S.tmem_base;
  bool bad = false;

  if (T == 0) {
    // nothing visible in this chunk: empty partial states
    if (threadIdx.x < nqv) {
      float* po = m.part_o + int64_t(it.part_base + threadIdx.x) * D;
      for (int c = 0; c < D; ++c) po[c] = 0.f;
      m.part_ml[it.part_base + threadIdx.x] = make_float2(-INFINITY, 0.f);
    }
    return;
  }

  if (warp == 0) {
    // ---------------- TMA producer ------------------------------------------
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      mbar_arrive_expect_tx(&S.q_full, 2 * kHalfBytes);
      tma_4d(S.q[0], &qmap, 0, 0, it.kv_head, it.row0, &S.q_full);
      tma_4d(S.q[1], &qmap, 64, 0, it.kv_head, it.row0, &S.q_full);
      const int32_t* pages = m.page_ids + m.page_indptr[it.lane];
      for (int j = 0; j < T && !bad; ++j) {
        const int st = j & 1;
        if (j >= 2 && !mbar_wait(&S.kv_empty[st], ((j >> 1) - 1) & 1)) {
          bad = true;
          break;
        }
        const int ts = kb + j * kTcTileSlots;
        const int te = min(ts + kTcTileSlots, ke);
        const int p0 = ts / P, p1 = (te - 1) / P;
        mbar_arrive_expect_tx(&S.kv_full[st], uint32_t(p1 - p0 + 1) * P * 128u * 4u);
        for (int pg = p0; pg <= p1; ++pg) {
          // first row of (page, kv head) in the [page * Hkv + head][slot] view
          const int yy = (pages[pg] * Hkv + it.kv_head) * P;
          const int off = (pg * P - ts) * 128;
#pragma unroll
          for (int a = 0; a < 2; ++a) {
            tma_2d(S.k[st][a] + off, &kmap, 64 * a, yy, &S.kv_full[st], pol);
            tma_2d(S.v[st][a] + off, &vmap, 64 * a, yy, &S.kv_full[st], pol);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ---------------------------------------------
    if (lane == 0) {
      constexpr uint32_t ID_S = idesc(128, 128, false);
      constexpr uint32_t ID_O = idesc(128, 128, true);
      const uint32_t tO = tmem + 256;
      auto pv = [&](int i) -> bool {
        const int st = i & 1;
        if (!mbar_wait(&S.p_full, i & 1)) return false;
        fence_after();
        const int valid = min(kTcTileSlots, ke - (kb + i * kTcTileSlots));
        const int ksteps = (valid + 15) >> 4;
        for (int k = 0; k < ksteps; ++k) {
          const uint64_t a = sdesc(S.p[k >> 2] + (k & 3) * 32, 16, 1024);
          const uint64_t b = sdesc(S.v[st][0] + k * 2048, kHalfBytes, 1024);
          mma(tO, a, b, ID_O, (i > 0 || k > 0) ? 1u : 0u);
        }
        commit(&S.o_done);
        commit(&S.kv_empty[st]);
        return true;
      };
      if (!mbar_wait(&S.q_full, 0)) bad = true;
      for (int j = 0; j < T && !bad; ++j) {
        const int st = j & 1, b = j & 1;
        if (!mbar_wait(&S.kv_full[st], (j >> 1) & 1)) { bad = true; break; }
        if (j >= 2 && !mbar_wait(&S.s_free[b], ((j >> 1) - 1) & 1)) { bad = true; break; }
        fence_after();
        const uint32_t tS = tmem + b * 128;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t a = sdesc(S.q[k >> 2] + (k & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc(S.k[st][k >> 2] + (k & 3) * 32, 16, 1024);
          mma(tS, a, bd, ID_S, k > 0 ? 1u : 0u);
        }
        commit(&S.s_full[b]);
        if (j >= 1 && !pv(j - 1)) { bad = true; break; }
      }
      if (!bad && !pv(T - 1)) bad = true;
    }
  } else {
    // ---------------- softmax warps (one query row per thread) --------------
    const int quad = warp & 3;
    const int qm = quad * 32 + lane;  // query index == TMEM lane
    const bool valid_q = qm < nqv;
    const int row = it.row0 + (valid_q ? qm : 0) / G;
    const int row_slot = valid_q ? m.slots[row] : -1;
    const int64_t mbase = (mask_words && valid_q) ? m.mask_word_indptr[row] : 0;
    const uint32_t tl = tmem + (uint32_t(quad * 32) << 16);
    float m_run = -INFINITY, l_run = 0.f;
    float s[128];
    for (int j = 0; j < T; ++j) {
      const int b = j & 1;
      const int ts = kb + j * kTcTileSlots;
      uint32_t words[4] = {0u, 0u, 0u, 0u};
      if (mask_words && valid_q) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (ts + 32 * i < ke) words[i] = mask_words[mbase + (ts >> 5) + i];
      }
      if (!mbar_wait(&S.s_full[b], (j >> 1) & 1)) { bad = true; break; }
      fence_after();
      tmem_ld128(tl + b * 128, s);
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.s_free[b]);
      float tmax = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; ++c) {
        const int sa = ts + c;
        const bool vis = valid_q && sa < ke &&
                         (mask_words ? ((words[c >> 5] >> (c & 31)) & 1u) != 0 : sa <= row_slot);
        s[c] = vis ? s[c] * scale_log2 : -INFINITY;
        tmax = fmaxf(tmax, s[c]);
      }
      const float m_new = fmaxf(m_run, tmax);
      const bool none = m_new == -INFINITY;
      const float alpha = none ? 1.f : exp2f(m_run - m_new);
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < 128; ++c) {
        const float p = none ? 0.f : exp2f(s[c] - m_new);
        s[c] = p;
        rs += p;
      }
      l_run = l_run * alpha + rs;
      m_run = m_new;
      // P.V of the previous tile must be done: it reads the P buffer and
      // accumulates into O, both of which change below
      if (j >= 1) {
        if (!mbar_wait(&S.o_done, (j - 1) & 1)) { bad = true; break; }
        fence_after();
      }
      // P row -> shared memory, bf16, 128-byte swizzle: [slot half][query][128 B]
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint8_t* rowp = S.p[h] + qm * 128;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            __nv_bfloat162 v2 = __floats2bfloat162_rn(s[h * 64 + ch * 8 + 2 * e],
                                                      s[h * 64 + ch * 8 + 2 * e + 1]);
            w[e] = *reinterpret_cast<uint32_t*>(&v2);
          }
          *reinterpret_cast<uint4*>(rowp + ((ch ^ (qm & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
        float o[128];
        tmem_ld128(tl + 256, o);
#pragma unroll
        for (int c = 0; c < 128; ++c) o[c] *= alpha;
        tmem_st128(tl + 256, o);
      }
      // last tile: zero the V rows between the last valid slot and the end of
      // its 16-slot MMA step (they hold whatever the page held past kv_len)
      const int valid = min(kTcTileSlots, ke - ts);
      if (j == T - 1 && (valid & 15)) {
        const int r0 = valid, r1 = (valid + 15) & ~15;
        const int chunks = (r1 - r0) * 8 * 2;
        for (int i = threadIdx.x - 64; i < chunks; i += 128) {
          const int h = i / ((r1 - r0) * 8), rem = i % ((r1 - r0) * 8);
          *reinterpret_cast<uint4*>(S.v[j & 1][h] + (r0 + rem / 8) * 128 + (rem % 8) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.p_full);
    }
    if (!bad && !mbar_wait(&S.o_done, (T - 1) & 1)) bad = true;
    fence_after();
    float o[128];
    tmem_ld128(tl + 256, o);
    if (valid_q && !bad) {
      float4* po = reinterpret_cast<float4*>(m.part_o + int64_t(it.part_base + qm) * D);
#pragma unroll
      for (int c = 0; c < 32; ++c) po[c] = make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
      m.part_ml[it.part_base + qm] = make_float2(m_run, l_run);
    }
  }
  if (bad) set_status(status, PIE_STATUS_TIMEOUT);
  fence_before();
  __syncthreads();
  if (warp == 1) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------
// host side: tensor maps and launch
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

static bool make_map(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
                     const cuuint64_t* strides, const cuuint32_t* box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_attend_tc(const pie_fwd_plan_t& p, const void* q_rot, const void* k_pool,
                             const void* v_pool, const uint32_t* mask_words, uint32_t* status,
                             cudaStream_t s) {
  const int D = p.desc.head_dim, Hq = p.desc.num_q_heads, Hkv = p.desc.num_kv_heads;
  const int G = p.G, P = p.desc.page_size;
  if (D != 128 || p.desc.dtype != PIE_BF16) return cudaErrorNotSupported;
  CUtensorMap qm, km, vm;
  {
    const cuuint64_t dims[4] = {cuuint64_t(D), cuuint64_t(G), cuuint64_t(Hkv), cuuint64_t(p.N)};
    const cuuint64_t str[3] = {cuuint64_t(D) * 2, cuuint64_t(G) * D * 2, cuuint64_t(Hq) * D * 2};
    const cuuint32_t box[4] = {64, cuuint32_t(G), 1, cuuint32_t(kTcTileQueries / G)};
    if (!make_map(&qm, q_rot, 4, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {cuuint64_t(D), cuuint64_t(p.num_pool_pages) * Hkv * P};
    const cuuint64_t str[1] = {cuuint64_t(D) * 2};
    const cuuint32_t box[2] = {64, cuuint32_t(P)};
    if (!make_map(&km, k_pool, 2, dims, str, box)) return cudaErrorInvalidValue;
    if (!make_map(&vm, v_pool, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  const size_t smem = sizeof(tc::Smem) + 1024;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attend_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  attend_tc_kernel<<<p.num_tc_items, tc::kThreads, smem, s>>>(
      p.dev, G, Hkv, P, p.desc.sm_scale * 1.4426950408889634f, mask_words, status, qm, km, vm);
  return cudaGetLastError();
}

}  // namespace pie
