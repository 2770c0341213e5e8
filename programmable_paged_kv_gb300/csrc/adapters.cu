// Per-lane adapters at a projection site (Pie "The forward pass", section
// Adapters).  Every row of lane l takes the lane's adapter a: a LoRA pair
// A_a [r][d_in], B_a [d_out][r] with a scale c_a, and an optional IA3 vector
// s_a [d_out]:
//     y' = (y + c_a B_a (A_a x)) * s_a          (elementwise in s_a)
// written over y in place; rows of lanes without an adapter keep y.
//
// The rows are cut into tiles of up to 128 consecutive rows of one lane
// (planned once per pass, reused at every site and layer), and each site
// runs two kernels:
//   shrink  t = A_a x on the tensor cores.  The adapter's rank is the MMA's
//           M side and the tile's rows its N side (rounded up to 16), so a
//           one-row decode lane costs a 16-column tile, not a 128-row one.
//           A_a fills the first r of the 128 operand rows; the rows after it
//           read whatever follows in shared memory, and their accumulator
//           lanes are never read.  A CTA covers one range of d_in for one
//           tile: warp 0 streams 64-column chunks of A_a and of the tile's x
//           rows (2-D tensor maps, 128-byte swizzle, each box copied from its
//           own lane) through a 4-deep ring, one thread of warp 1 issues four
//           K=16 MMAs per chunk into a TMEM accumulator [r lanes x N
//           columns], and the first r/32 warps store the fp32 partial sums of
//           their range.
//   expand  y' = (y + c_a B_a t) * s_a on the CUDA cores in fp32: one CTA per
//           (tile, 256 output columns), one column per thread.  The tile's y
//           rows arrive by 1-D bulk copies in groups of 16 rows, t (the
//           partial sums added up and scaled by c_a) sits in shared memory,
//           each thread keeps its column's row of B_a in registers, and every
//           finished group goes back to y by bulk stores.
// The expand moves 4 bytes of y per output for r multiply-adds and is bound
// by HBM, so it stays off the tensor cores; the shrink does r multiply-adds
// per 2 bytes of x, the contraction that needs them.  Every wait is bounded
// in time (PIE_STATUS_TIMEOUT).
//
// Plans whose adapters each serve few rows (decode: a row per lane) take one
// kernel instead, grouped by adapter: a cluster of 8 CTAs per adapter in use.
// CTA c forms the rank-r partial sums of the group's rows over its eighth of
// d_in (CUDA cores, fp32), the cluster adds the eight partials up through
// distributed shared memory, and CTA c applies y' = (y + c_a B_a t) * s_a to
// its eighth of d_out, with its B_a rows and y values loaded before the
// exchange.  Two kernels and the partial sums' round trip through global
// memory would cost more than the whole of this work.

#include <algorithm>
#include <cstring>
#include <vector>

#include <cooperative_groups.h>

#include "internal.h"
#include "tc_util.cuh"

namespace pie {
namespace ad {

constexpr int kTileRows = 128;   // rows per tile (the MMA's largest N used here)
constexpr int kChunk = 64;       // d_in columns per ring stage: one 128-byte swizzle row
constexpr int kStages = 6;       // shrink ring depth
constexpr int kMaxSplits = 8;    // d_in ranges per tile (partial sums kept per range)
constexpr int kOBlock = 256;     // output columns per expand CTA
constexpr int kExpandThreads = 256;  // one output column (TMEM lane) per thread
constexpr int kGroupRows = 16;   // y rows per arrival barrier in the expand
constexpr int kMaxGroups = kTileRows / kGroupRows;
constexpr int kShrinkCtasPerSm = 3;
static_assert(kMaxGroups * 8 <= 128, "expand barriers live in the first 128 bytes");

// Up to kTileRows consecutive rows [row0, row0 + n) of one lane and its adapter.
struct alignas(16) Tile {
  int32_t row0, n, adapter, pad;
};

// Shrink shared memory, laid out for the plan's largest tile (nmax rows):
// a 1 KB header, then kStages A_a chunks (R rows x 64 columns, bf16), then
// kStages x chunks (nmax rows x 64 columns), then a guard so that the M=128
// operand read from the last A stage (128 rows) stays inside the allocation.
struct ShrinkHdr {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t done;
  uint32_t tmem_base;
  int last;  // this CTA is the tile's last d_in range to finish
};
static_assert(sizeof(ShrinkHdr) <= 1024, "shrink header");

__host__ __device__ constexpr size_t shrink_smem_bytes(int R, int nmax) {
  return 1024 + size_t(kStages) * R * 128 + size_t(kStages) * nmax * 128 +
         (size_t(kStages) * nmax * 128 + size_t(R) * 128 < 128 * 128
              ? 128 * 128 - size_t(kStages) * nmax * 128 - size_t(R) * 128
              : 0);
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 16 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* f) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];\n\ttcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) f[i] = __uint_as_float(r[i]);
}

// 1-D bulk copy shared -> global in the calling thread's bulk group.
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
               "r"(smem_u32(src)), "r"(bytes)
               : "memory");
}
// 2-D tensor store shared -> global (the map's box at {x, y}) in the calling
// thread's bulk group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y,
                                             const void* src) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map),
      "r"(x), "r"(y), "r"(smem_u32(src))
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

}  // namespace ad

// t[row][k] = c_a sum_i A_a[k][i] x[row][i] for the tile's rows.  With d_in cut
// into `splits` ranges, each CTA stores its range's sums to t_part[split] and
// the last CTA of the tile to finish adds them up in range order (the result
// does not depend on which CTA finishes last) and resets the tile's counter.
template <int R>
__global__ void __launch_bounds__(128) adapter_shrink_kernel(
    const ad::Tile* __restrict__ tiles, int splits, int chunks_per_split, int num_chunks,
    int num_rows, const float* scale, float* t_part, float* t_final, int* counters,
    uint32_t* status,
    int nmax, uint32_t tmem_cols, const __grid_constant__ CUtensorMap xmap,
    const __grid_constant__ CUtensorMap amap) {
  using namespace ad;
  using namespace tc;
  extern __shared__ uint8_t raw_[];
  uint8_t* raw = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw_) + 1023) &
                                            ~uintptr_t(1023));
  ShrinkHdr& S = *reinterpret_cast<ShrinkHdr*>(raw);
  uint8_t* a_st = raw + 1024;                       // stage st at a_st + st * R * 128
  uint8_t* x_st = a_st + size_t(kStages) * R * 128;  // stage st at x_st + st * nmax * 128
  const Tile tile = tiles[blockIdx.x];
  const int split = blockIdx.y;
  const int c0 = split * chunks_per_split;
  const int nc = min(num_chunks, c0 + chunks_per_split) - c0;  // >= 1 (host sizing)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = (tile.n + 15) & ~15;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    mbar_init(&S.done, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&S.tmem_base)),
                 "r"(tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = S.tmem_base;
  // after the kernels before it (x is read below); every CTA of this grid
  // holds its TMEM now: the expand kernel may start its set-up (it waits for
  // this grid before it reads A x)
  grid_dep_wait();
  grid_dep_launch();
  bool bad = false;

  if (warp == 0) {
    // ---- producer: lane i < N/16 copies x rows [row0 + 16 i, +16), lane 31 A_a
    const uint64_t pol_x = policy_evict_first();
    const uint64_t pol_a = policy_evict_last();
    int issued = 0;
    for (int i = 0; i < nc; ++i) {
      const int st = i % kStages;
      if (i >= kStages) {
        int ok = lane == 0 ? int(mbar_wait(&S.empty[st], ((i / kStages) - 1) & 1)) : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          bad = true;
          break;
        }
      }
      if (lane == 0) mbar_arrive_expect_tx(&S.full[st], uint32_t(R + N) * 128u);
      __syncwarp();
      const int cx = (c0 + i) * kChunk;
      if (lane < N / 16)
        tma_2d(x_st + size_t(st) * nmax * 128 + lane * 2048, &xmap, cx, tile.row0 + lane * 16,
               &S.full[st], pol_x);
      if (lane == 31) tma_2d(a_st + st * R * 128, &amap, cx, tile.adapter * R, &S.full[st], pol_a);
      issued = i + 1;
    }
    // copies still in flight must land before the CTA may exit
    if (lane == 0)
      for (int i = max(0, issued - kStages); i < issued; ++i)
        if (!mbar_wait(&S.full[i % kStages], (i / kStages) & 1)) bad = true;
    __syncwarp();
  } else if (warp == 1) {
    // ---- MMA issuer: D[k][j] += A_a[k][c] x[j][c] over the chunk, 4 x K=16
    if (lane == 0) {
      const uint32_t id = idesc(128, N, false);
      for (int i = 0; i < nc; ++i) {
        const int st = i % kStages;
        if (!mbar_wait(&S.full[st], (i / kStages) & 1)) {
          bad = true;
          break;
        }
        fence_after();
        const uint64_t da = sdesc(a_st + st * R * 128, 16, 1024);
        const uint64_t dx = sdesc(x_st + size_t(st) * nmax * 128, 16, 1024);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ss(tmem, da + 2 * k, dx + 2 * k, id, (i > 0 || k > 0) ? 1u : 0u);
        commit(&S.empty[st]);
      }
      commit(&S.done);  // arrives when every MMA issued above has completed
    }
    __syncwarp();
  }

  // ---- epilogue: TMEM lane k holds t[row0 + j][k] at column j
  if (warp < (R + 31) / 32) {
    int ok = lane == 0 ? int(mbar_wait(&S.done, 0)) : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
      bad = true;
    } else {
      fence_after();
      const int k = warp * 32 + lane;
      const float c = splits == 1 ? scale[tile.adapter] : 1.f;
      float* dst = (splits == 1 ? t_final + int64_t(tile.row0) * R
                                : t_part + (int64_t(split) * num_rows + tile.row0) * R) + k;
      for (int cb = 0; cb < N; cb += 16) {
        float v[16];
        tmem_ld16(tmem + (uint32_t(warp * 32) << 16) + uint32_t(cb), v);
        if (k < R) {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj)
            if (cb + jj < tile.n) dst[int64_t(cb + jj) * R] = v[jj] * c;
        }
      }
      __threadfence();  // this range's sums are visible before the counter moves
    }
  }
  if (splits > 1) {
    __syncthreads();
    if (threadIdx.x == 0) S.last = atomicAdd(&counters[blockIdx.x], 1) == splits - 1;
    __syncthreads();
    if (S.last) {
      __threadfence();
      const float c = scale[tile.adapter];
      const int cnt = tile.n * R;
      const float* src0 = t_part + int64_t(tile.row0) * R;
      constexpr int kBatch = 4;  // elements per thread whose loads are in flight together
      for (int e0 = threadIdx.x; e0 < cnt; e0 += 128 * kBatch) {
        float p[kBatch][kMaxSplits];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          const int e = e0 + 128 * b;
#pragma unroll
          for (int q = 0; q < kMaxSplits; ++q)
            p[b][q] = (q < splits && e < cnt) ? __ldcg(src0 + int64_t(q) * num_rows * R + e) : 0.f;
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          const int e = e0 + 128 * b;
          float acc = 0.f;
#pragma unroll
          for (int q = 0; q < kMaxSplits; ++q) acc += p[b][q];
          if (e < cnt) t_final[int64_t(tile.row0) * R + e] = acc * c;
        }
      }
      if (threadIdx.x == 0) counters[blockIdx.x] = 0;  // ready for the next apply
    }
  }
  if (bad) set_status(status, PIE_STATUS_TIMEOUT);
  fence_before();
  __syncthreads();
  if (warp == 1) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(tmem_cols)
                 : "memory");
  }
}

namespace ad {

// Expand operand geometry for rank R: t is split into bf16 parts hi + lo (t
// to about 16 bits); the MMA's K runs over [hi | lo], each part padded to a
// multiple of 16, in 128-byte swizzled K halves (one half up to rank 32).
template <int R>
struct ExpandCfg {
  static constexpr int KP = R < 16 ? 16 : R;   // one part, padded to a K step
  static constexpr int H = (2 * KP + 63) / 64;  // 128-byte K halves
  static constexpr int KSTEPS = 2 * KP / 16;    // K=16 MMAs per 128 output columns
};

// Byte offset of element (row, k) in a K-major operand of `rows` rows laid out
// as H halves of 64 K columns, 128-byte swizzle (8-row atoms of 1024 bytes).
__device__ __forceinline__ uint32_t sw128_offset(int rows, int row, int k) {
  const int half = k >> 6, c = (k & 63) >> 3;
  return uint32_t(half * rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 +
                  ((c ^ (row & 7)) << 4) + ((k & 7) << 1));
}

}  // namespace ad

// y[row][o] = (y[row][o] + sum_k B_a[o][k] t[row][k]) * s_a[o] for the tile's
// rows and 256 output columns (t already scaled by c_a).  B_a t runs on the
// tensor cores: two M=128 tiles of output columns, N = the tile's rows rounded
// up to 16, K over [t_hi | t_lo]; each thread then owns one output column of
// one M tile (its TMEM lane) and streams the tile's y rows through shared
// memory, 16 rows (one tcgen05.ld) at a time.
template <int R>
__global__ void __launch_bounds__(ad::kExpandThreads) adapter_expand_kernel(
    const ad::Tile* __restrict__ tiles, const float* t_final,
    const __nv_bfloat16* __restrict__ lora_b, const __nv_bfloat16* __restrict__ ia3,
    __nv_bfloat16* y, int d_out, int max_rows, uint32_t tmem_cols,
    uint32_t* status, const __grid_constant__ CUtensorMap ymap) {
  using namespace ad;
  using namespace tc;
  using C = ExpandCfg<R>;
  extern __shared__ uint8_t raw_[];
  uint8_t* raw = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw_) + 1023) &
                                            ~uintptr_t(1023));
  const int nmax = (max_rows + 15) & ~15;
  const size_t ys_bytes = (size_t(max_rows) * kOBlock * 2 + 1023) & ~size_t(1023);
  const size_t a_bytes = R > 0 ? size_t(2) * C::H * 128 * 128 : 0;
  const size_t b_bytes = R > 0 ? size_t(C::H) * nmax * 128 : 0;
  __nv_bfloat16* ys = reinterpret_cast<__nv_bfloat16*>(raw);  // [max_rows][256]
  uint8_t* a_op = raw + ys_bytes;                              // [2][H][128 rows][128 B]
  uint8_t* b_op = a_op + a_bytes;                              // [H][nmax rows][128 B]
  uint64_t* bar = reinterpret_cast<uint64_t*>(b_op + b_bytes); // [kMaxGroups] y groups
  uint64_t* mma_done = bar + kMaxGroups;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

  const Tile tile = tiles[blockIdx.x];
  const int o0 = blockIdx.y * kOBlock;
  const int n = tile.n, a = tile.adapter;
  const int N = (n + 15) & ~15;
  const int ngroups = (n + kGroupRows - 1) / kGroupRows;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int g = 0; g < ngroups; ++g) mbar_init(&bar[g], 1);
    mbar_init(mma_done, 1);
    fence_barrier_init();
  }
  if constexpr (R > 0) {
    if (warp == 0) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(tmem_slot)),
                   "r"(tmem_cols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  fence_before();
  __syncthreads();
  fence_after();

  // full groups of 16 rows move as one 2-D box each way; the rows of a last,
  // partial group one by one (a box would also cover the next lane's rows)
  __nv_bfloat16* yt = y + int64_t(tile.row0) * d_out + o0;
  const int nfull = n / kGroupRows;
  if (warp == 0) {
    if (lane < ngroups)
      mbar_arrive_expect_tx(&bar[lane],
                            uint32_t(min(kGroupRows, n - lane * kGroupRows)) * kOBlock * 2u);
    __syncwarp();
    if (lane < nfull)
      tma_2d(ys + lane * kGroupRows * kOBlock, &ymap, o0, tile.row0 + lane * kGroupRows,
             &bar[lane], policy_evict_first());
    for (int j = nfull * kGroupRows + lane; j < n; j += 32)
      bulk_g2s(ys + j * kOBlock, yt + int64_t(j) * d_out, kOBlock * 2, &bar[j / kGroupRows]);
  }

  // this thread's output column: M tile m = warp / 4, TMEM lane quarter q
  const int m = warp >> 2, q = warp & 3;
  const int ol = m * 128 + q * 32 + lane;
  const float s_o = ia3 ? __bfloat162float(ia3[int64_t(a) * d_out + o0 + ol]) : 1.f;
  uint32_t tmem = 0;
  bool bad = false;

  if constexpr (R > 0) {
    // operands: A = B_a rows [o0, o0 + 256) as [hi copy | lo copy] of K, B = [t_hi | t_lo]
    constexpr int CH = R / 8;  // 16-byte chunks of one row of B_a or of t
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    for (int i = tid; i < kOBlock * CH; i += kExpandThreads) {
      const int row = i / CH, c = i % CH;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(
                                lora_b + (int64_t(a) * d_out + o0 + row) * R) + c);
      uint8_t* base = a_op + (row >> 7) * (C::H * 128 * 128);
      const int r = row & 127;
      *reinterpret_cast<uint4*>(base + sw128_offset(128, r, 8 * c)) = v;
      *reinterpret_cast<uint4*>(base + sw128_offset(128, r, C::KP + 8 * c)) = v;
      if (R < C::KP) {  // zero K padding of both parts
        *reinterpret_cast<uint4*>(base + sw128_offset(128, r, R + 8 * c)) = zero;
        *reinterpret_cast<uint4*>(base + sw128_offset(128, r, C::KP + R + 8 * c)) = zero;
      }
    }
    // y, B_a and the IA3 scale above were written before the shrink kernel
    // started; A x is the shrink kernel's
    grid_dep_wait();
    const float* tsrc = t_final + int64_t(tile.row0) * R;
    for (int i = tid; i < n * CH; i += kExpandThreads) {
      const int j = i / CH, c = i % CH;
      const float4 f0 = __ldcg(reinterpret_cast<const float4*>(tsrc + j * R + 8 * c));
      const float4 f1 = __ldcg(reinterpret_cast<const float4*>(tsrc + j * R + 8 * c + 4));
      const float f[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * e], f[2 * e + 1]);
        const __nv_bfloat162 l = __floats2bfloat162_rn(f[2 * e] - __low2float(h),
                                                       f[2 * e + 1] - __high2float(h));
        hi[e] = *reinterpret_cast<const uint32_t*>(&h);
        lo[e] = *reinterpret_cast<const uint32_t*>(&l);
      }
      *reinterpret_cast<uint4*>(b_op + sw128_offset(nmax, j, 8 * c)) =
          make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(b_op + sw128_offset(nmax, j, C::KP + 8 * c)) =
          make_uint4(lo[0], lo[1], lo[2], lo[3]);
      if (R < C::KP) {
        *reinterpret_cast<uint4*>(b_op + sw128_offset(nmax, j, R + 8 * c)) = zero;
        *reinterpret_cast<uint4*>(b_op + sw128_offset(nmax, j, C::KP + R + 8 * c)) = zero;
      }
    }
    fence_proxy_async_smem();  // generic-proxy writes, read by the tensor cores
    fence_before();
    __syncthreads();
    fence_after();
    tmem = *tmem_slot;
    if (tid == 0) {
      const uint32_t id = idesc(128, N, false);
      const uint64_t db = sdesc(b_op, 16, 1024);
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const uint64_t da = sdesc(a_op + mt * (C::H * 128 * 128), 16, 1024);
#pragma unroll
        for (int ks = 0; ks < C::KSTEPS; ++ks) {
          const uint64_t offa = uint64_t((ks >> 2) * ((128 * 128) >> 4) + (ks & 3) * 2);
          const uint64_t offb = uint64_t((ks >> 2) * ((nmax * 128) >> 4) + (ks & 3) * 2);
          mma_ss(tmem + uint32_t(mt * nmax), da + offa, db + offb, id, ks > 0 ? 1u : 0u);
        }
      }
      commit(mma_done);
    }
    const bool ok = mbar_wait(mma_done, 0);
    if (__syncthreads_or(!ok)) bad = true;
    fence_after();
  } else {
    __syncthreads();
  }

  for (int g = 0; g < ngroups && !bad; ++g) {
    const bool ok = mbar_wait(&bar[g], 0);
    if (__syncthreads_or(!ok)) {
      bad = true;
      break;
    }
    const int j0 = g * kGroupRows, j1 = min(n, j0 + kGroupRows);
    float d[16];
    if constexpr (R > 0) {
      tmem_ld16(tmem + (uint32_t(q * 32) << 16) + uint32_t(m * nmax + j0), d);
    } else {
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) d[jj] = 0.f;
    }
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) {
      if (j0 + jj < j1) {
        __nv_bfloat16& yv = ys[(j0 + jj) * kOBlock + ol];
        yv = __float2bfloat16_rn((__bfloat162float(yv) + d[jj]) * s_o);
      }
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (g < nfull) {
      if (tid == 0) {
        tma_store_2d(&ymap, o0, tile.row0 + j0, ys + j0 * kOBlock);
        bulk_commit();
      }
    } else if (warp == 0 && lane < j1 - j0) {
      const int j = j0 + lane;
      bulk_s2g(yt + int64_t(j) * d_out, ys + j * kOBlock, kOBlock * 2);
      bulk_commit();
    }
  }
  if (warp == 0) bulk_wait_read_all();  // shared memory must outlive the stores' reads
  if (bad && tid == 0) {
    set_status(status, PIE_STATUS_TIMEOUT);
    for (int g = 0; g < ngroups; ++g) mbar_wait(&bar[g], 0);  // copies still in flight land first
  }
  if constexpr (R > 0) {
    fence_before();
    __syncthreads();
    if (warp == 0) {
      fence_after();
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                   "r"(tmem_cols)
                   : "memory");
    }
  }
}


// ---------------------------------------------------------------------------
// Grouped adapters for few rows per adapter: one cluster of kGCluster CTAs
// per adapter in use (see the top of this file).
// ---------------------------------------------------------------------------
namespace ad {

constexpr int kGCluster = 8;      // CTAs per adapter: d_in and d_out cut in eighths
constexpr int kGMaxRows = 16;     // rows an adapter may serve on this path
constexpr int kGThreads = 256;

// An adapter in use and its rows: rows[row_off .. row_off + n).
struct alignas(16) Group {
  int32_t row_off, n, adapter, pad;
};

}  // namespace ad

template <int R, int NR>
__global__ void __cluster_dims__(ad::kGCluster, 1, 1) __launch_bounds__(ad::kGThreads)
    adapter_group_kernel(const ad::Group* __restrict__ groups, const int32_t* __restrict__ rows,
                         int d_in, int d_out, const __nv_bfloat16* __restrict__ x,
                         __nv_bfloat16* y, const __nv_bfloat16* __restrict__ lora_a,
                         const __nv_bfloat16* __restrict__ lora_b,
                         const float* __restrict__ scale, const __nv_bfloat16* __restrict__ ia3) {
  using namespace ad;
  namespace cg = cooperative_groups;
  constexpr int kWarps = kGThreads / 32;
  constexpr int KPW = (R + kWarps - 1) / kWarps;  // ranks per warp
  cg::cluster_group cluster = cg::this_cluster();
  const int c = int(cluster.block_rank());
  const Group g = groups[blockIdx.x / kGCluster];
  const int n = g.n, a = g.adapter;  // n <= NR
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  __shared__ float part[NR * R];  // this CTA's partial sums
  __shared__ float tot[NR * R];   // the cluster's, scaled by c_a
  int my_rows[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) my_rows[r] = rows[g.row_off + (r < n ? r : 0)];
  // this CTA's eighth of d_in, in 16-byte vectors of x and A; a lane takes
  // vectors lane, lane + 32, ... of it
  const int units = d_in / 8;
  const int u0 = c * units / kGCluster, u1 = (c + 1) * units / kGCluster;

  // the expand's operands first (they do not depend on the exchange): this
  // thread's first pair of output columns, its B_a rows (bf16 pairs) and y
  const int ncols = d_out / kGCluster, col0 = c * ncols, pairs = ncols / 2;
  const __nv_bfloat16* Ba = lora_b + int64_t(a) * d_out * R;
  uint32_t bq[2][R / 2];
  __nv_bfloat162 yq[NR];
  auto load_pair = [&](int cp) {
    const int o = col0 + 2 * cp;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint4* src = reinterpret_cast<const uint4*>(Ba + int64_t(o + k) * R);
#pragma unroll
      for (int v = 0; v < R / 8; ++v) {
        const uint4 u = src[v];
        bq[k][4 * v] = u.x;
        bq[k][4 * v + 1] = u.y;
        bq[k][4 * v + 2] = u.z;
        bq[k][4 * v + 3] = u.w;
      }
    }
#pragma unroll
    for (int r = 0; r < NR; ++r)
      yq[r] = *reinterpret_cast<const __nv_bfloat162*>(y + int64_t(my_rows[r]) * d_out + o);
  };
  if (tid < pairs) load_pair(tid);

  // shrink: warp w takes ranks w, w + 8, ... in passes of KB ranks (at most
  // 32 (rank, row) accumulator pairs live); per step of 32 vectors the A_a
  // and x vectors of the pass's ranks and all rows are loaded together, then
  // one dot product per (rank, row) is reduced across the warp.  Rows past n
  // repeat the first row (finite) and are never stored.
  constexpr int KB = (32 / NR) < KPW ? (32 / NR < 1 ? 1 : 32 / NR) : KPW;
  const uint4* Aa = reinterpret_cast<const uint4*>(lora_a + int64_t(a) * R * d_in);
#pragma unroll 1
  for (int i0 = 0; i0 < KPW; i0 += KB) {
    float acc[KB][NR], acc2[KB][NR];  // even and odd elements (one packed FMA)
#pragma unroll
    for (int i = 0; i < KB; ++i)
#pragma unroll
      for (int r = 0; r < NR; ++r) acc[i][r] = acc2[i][r] = 0.f;
    for (int u = u0 + lane; u < u1; u += 32) {
      uint4 av[KB], xv[NR];
#pragma unroll
      for (int i = 0; i < KB; ++i) {
        const int k = warp + kWarps * (i0 + i);
        av[i] = k < R ? Aa[int64_t(k) * units + u] : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int r = 0; r < NR; ++r)
        xv[r] = reinterpret_cast<const uint4*>(x + int64_t(my_rows[r]) * d_in)[u];
#pragma unroll
      for (int i = 0; i < KB; ++i) {
        float af[8];
        unpack16<__nv_bfloat16>(av[i], af);
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          float xf[8];
          unpack16<__nv_bfloat16>(xv[r], xf);
#pragma unroll
          for (int e = 0; e < 8; e += 2)
            ffma2(acc[i][r], acc2[i][r], af[e], af[e + 1], xf[e], xf[e + 1], acc[i][r], acc2[i][r]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < KB; ++i) {
      const int k = warp + kWarps * (i0 + i);
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        float v = acc[i][r] + acc2[i][r];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0 && k < R && r < n) part[r * R + k] = v;
      }
    }
  }
  // the cluster's eight partials, summed and scaled by c_a, in every CTA
  cluster.sync();
  const float ca = scale[a];
  for (int i = tid; i < n * R; i += kGThreads) {
    float v = 0.f;
#pragma unroll
    for (int q = 0; q < kGCluster; ++q) v += cluster.map_shared_rank(part, q)[i];
    tot[i] = v * ca;
  }
  // no CTA leaves, and with it its shared memory, before every peer has read it
  cluster.sync();

  // expand: y' = (y + c_a B_a t) * s_a over this CTA's columns, two per thread
  for (int cp = tid; cp < pairs; cp += kGThreads) {
    if (cp != tid) load_pair(cp);
    const int o = col0 + 2 * cp;
    float s0 = 1.f, s1 = 1.f;
    if (ia3) {
      s0 = __bfloat162float(ia3[int64_t(a) * d_out + o]);
      s1 = __bfloat162float(ia3[int64_t(a) * d_out + o + 1]);
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      if (r < n) {
        float d0 = 0.f, d1 = 0.f;
        const float* tr = tot + r * R;
#pragma unroll
        for (int k = 0; k < R / 2; ++k) {
          const float t0 = tr[2 * k], t1 = tr[2 * k + 1];
          const uint32_t b0 = bq[0][k], b1 = bq[1][k];
          d0 = fmaf(t0, __uint_as_float(b0 << 16), d0);
          d0 = fmaf(t1, __uint_as_float(b0 & 0xFFFF0000u), d0);
          d1 = fmaf(t0, __uint_as_float(b1 << 16), d1);
          d1 = fmaf(t1, __uint_as_float(b1 & 0xFFFF0000u), d1);
        }
        const float2 yv = __bfloat1622float2(yq[r]);
        *reinterpret_cast<__nv_bfloat162*>(y + int64_t(my_rows[r]) * d_out + o) =
            __floats2bfloat162_rn((yv.x + d0) * s0, (yv.y + d1) * s1);
      }
    }
  }
}

}  // namespace pie

// ---------------------------------------------------------------------------
// host side: plan and launches
// ---------------------------------------------------------------------------
struct pie_fwd_adapter_plan {
  int32_t num_lanes, num_rows, num_adapters, max_rank;
  int32_t num_tiles, max_tile_rows;
  pie::ad::Tile* tiles;  // device, in the workspace
  int* counters;         // device: finished d_in ranges per tile (zero between applies)
  float* t_part;         // device scratch: [kMaxSplits][num_rows][rank] partial sums
  float* t_final;        // device scratch: [num_rows][rank], c_a A_a x
  // grouped path (every adapter serves at most kGMaxRows rows): one cluster
  // per adapter in use; num_groups 0 when the plan does not take it
  int32_t num_groups, max_group_rows;
  pie::ad::Group* groups;  // device, in the workspace
  int32_t* group_rows;     // device: the groups' rows
  pie::PinnedBlock* staging;
};

namespace {

using pie::set_last_error;

int check_lanes(int32_t num_lanes, const int32_t* row_indptr, int64_t* num_tiles) {
  if (num_lanes < 0) return set_last_error(PIE_EINVAL, "num_lanes < 0");
  if (!row_indptr) return set_last_error(PIE_EINVAL, "row_indptr is NULL");
  if (row_indptr[0] != 0) return set_last_error(PIE_EINVAL, "row_indptr[0] != 0");
  int64_t t = 0;
  for (int l = 0; l < num_lanes; ++l) {
    if (row_indptr[l + 1] < row_indptr[l])
      return set_last_error(PIE_EINVAL, "row_indptr is not monotone");
    t += (int64_t(row_indptr[l + 1]) - row_indptr[l] + pie::ad::kTileRows - 1) /
         pie::ad::kTileRows;
  }
  *num_tiles = t;
  return PIE_OK;
}

bool rank_built(int r) { return r == 0 || r == 8 || r == 16 || r == 32 || r == 64; }

// workspace: tiles | counters (both uploaded, counters as zeros) | t_part | t_final
struct WsLayout {
  size_t tiles = 0, counters = 0, groups = 0, group_rows = 0, t_part = 0, t_final = 0, total = 0;
};

// tiles, per-tile counters, groups (at most one per tile) and their rows are
// uploaded in one copy; the partial sums follow
WsLayout ws_layout(int64_t num_tiles, int64_t num_rows, int max_rank) {
  auto up = [](size_t v) { return (v + 255) & ~size_t(255); };
  WsLayout Y;
  Y.tiles = 0;
  Y.counters = up(size_t(num_tiles) * sizeof(pie::ad::Tile));
  Y.groups = Y.counters + up(size_t(num_tiles) * 4);
  Y.group_rows = Y.groups + up(size_t(num_tiles) * sizeof(pie::ad::Group));
  Y.t_part = Y.group_rows + up(size_t(num_rows) * 4);
  Y.t_final =
      Y.t_part + up(size_t(pie::ad::kMaxSplits) * size_t(num_rows) * size_t(max_rank) * 4);
  Y.total = Y.t_final + up(size_t(num_rows) * size_t(max_rank) * 4);
  return Y;
}

template <int R>
cudaError_t launch_adapter(const pie_fwd_adapter_plan_t& p, int d_in, int d_out, const void* x,
                           void* y, const void* lora_a, const void* lora_b, const float* scale,
                           const void* ia3, uint32_t* status, cudaStream_t s) {
  using namespace pie;
  if constexpr (R > 0) {
    if (p.num_groups > 0) {
      // few rows per adapter: one kernel, a cluster per adapter in use, its
      // row loops sized for the plan's largest group
      auto go = [&](auto kernel) {
        kernel<<<p.num_groups * ad::kGCluster, ad::kGThreads, 0, s>>>(
            p.groups, p.group_rows, d_in, d_out, static_cast<const __nv_bfloat16*>(x),
            static_cast<__nv_bfloat16*>(y), static_cast<const __nv_bfloat16*>(lora_a),
            static_cast<const __nv_bfloat16*>(lora_b), scale,
            static_cast<const __nv_bfloat16*>(ia3));
        return cudaGetLastError();
      };
      if (p.max_group_rows <= 4) return go(adapter_group_kernel<R, 4>);
      if (p.max_group_rows <= 8) return go(adapter_group_kernel<R, 8>);
      return go(adapter_group_kernel<R, ad::kGMaxRows>);
    }
  }
  int splits = 1;
  if constexpr (R > 0) {
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int num_chunks = d_in / ad::kChunk;
    const int64_t want = (int64_t(ad::kShrinkCtasPerSm) * sms + p.num_tiles - 1) / p.num_tiles;
    splits = int(std::max<int64_t>(1, std::min<int64_t>(want, std::min(ad::kMaxSplits, num_chunks))));
    const int cps = (num_chunks + splits - 1) / splits;
    splits = (num_chunks + cps - 1) / cps;

    CUtensorMap xmap, amap;
    {
      const cuuint64_t dims[2] = {cuuint64_t(d_in), cuuint64_t(p.num_rows)};
      const cuuint64_t str[1] = {cuuint64_t(d_in) * 2};
      const cuuint32_t box[2] = {ad::kChunk, 16};
      if (!tc::make_map(&xmap, x, 2, dims, str, box)) return cudaErrorInvalidValue;
    }
    {
      const cuuint64_t dims[2] = {cuuint64_t(d_in), cuuint64_t(p.num_adapters) * R};
      const cuuint64_t str[1] = {cuuint64_t(d_in) * 2};
      const cuuint32_t box[2] = {ad::kChunk, cuuint32_t(R)};
      if (!tc::make_map(&amap, lora_a, 2, dims, str, box)) return cudaErrorInvalidValue;
    }
    const int nmax = (p.max_tile_rows + 15) & ~15;
    const size_t smem = 1024 + ad::shrink_smem_bytes(R, nmax);  // + alignment slack
    static std::atomic<uint64_t> configured{0};
    {
      cudaError_t e = set_smem_limit(adapter_shrink_kernel<R>,
                                     int(1024 + ad::shrink_smem_bytes(R, ad::kTileRows)), configured);
      if (e != cudaSuccess) return e;
    }
    uint32_t tmem_cols = 32;
    while (tmem_cols < uint32_t(nmax)) tmem_cols <<= 1;
    cudaError_t e = launch_dependent(adapter_shrink_kernel<R>, dim3(p.num_tiles, splits), dim3(128),
                                     smem, s, true, p.tiles, splits, cps, num_chunks, p.num_rows,
                                     scale, p.t_part, p.t_final, p.counters, status, nmax,
                                     tmem_cols, xmap, amap);
    if (e != cudaSuccess) return e;
  }
  // shared memory: 1 KB alignment slack, y rows, the two MMA operands, barriers
  using EC = ad::ExpandCfg<R>;
  auto expand_smem = [](int rows) {
    const size_t nmax = size_t((rows + 15) & ~15);
    const size_t ys = (size_t(rows) * ad::kOBlock * 2 + 1023) & ~size_t(1023);
    const size_t ops = R > 0 ? size_t(2) * EC::H * 128 * 128 + size_t(EC::H) * nmax * 128 : 0;
    return 1024 + ys + ops + 256;
  };
  const size_t smem = expand_smem(p.max_tile_rows);
  static std::atomic<uint64_t> configured_e{0};
  {
    cudaError_t e = set_smem_limit(adapter_expand_kernel<R>, int(expand_smem(ad::kTileRows)),
                                   configured_e);
    if (e != cudaSuccess) return e;
  }
  // TMEM: two M tiles of up to nmax columns, a power of two of at least 32
  uint32_t tmem_cols = 0;
  if (R > 0) {
    tmem_cols = 32;
    while (tmem_cols < uint32_t(2 * ((p.max_tile_rows + 15) & ~15))) tmem_cols <<= 1;
  }
  CUtensorMap ymap;
  {
    const cuuint64_t dims[2] = {cuuint64_t(d_out), cuuint64_t(p.num_rows)};
    const cuuint64_t str[1] = {cuuint64_t(d_out) * 2};
    const cuuint32_t box[2] = {ad::kOBlock, ad::kGroupRows};
    if (!tc::make_map(&ymap, y, 2, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  }
  // behind the shrink kernel (rank > 0) it starts while that one drains; with
  // no shrink kernel before it, in plain stream order
  return launch_dependent(adapter_expand_kernel<R>, dim3(p.num_tiles, d_out / ad::kOBlock),
                          dim3(ad::kExpandThreads), smem, s, R > 0, p.tiles, p.t_final,
                          static_cast<const __nv_bfloat16*>(lora_b),
                          static_cast<const __nv_bfloat16*>(ia3), static_cast<__nv_bfloat16*>(y),
                          d_out, p.max_tile_rows, tmem_cols, status, ymap);
}

}  // namespace

extern "C" {

int pie_fwd_adapter_workspace_bytes(int32_t num_lanes, const int32_t* row_indptr,
                                    int32_t max_rank, size_t* bytes) {
  if (!bytes) return set_last_error(PIE_EINVAL, "bytes is NULL");
  if (!rank_built(max_rank)) return set_last_error(PIE_EUNSUPPORTED, "max_rank not in {0, 8, 16, 32, 64}");
  int64_t nt = 0;
  int rc = check_lanes(num_lanes, row_indptr, &nt);
  if (rc != PIE_OK) return rc;
  *bytes = ws_layout(nt, row_indptr[num_lanes], max_rank).total;
  return PIE_OK;
}

int pie_fwd_adapter_plan(int32_t num_lanes, const int32_t* row_indptr,
                         const int32_t* adapter_of_lane, int32_t num_adapters, int32_t max_rank,
                         void* dev_workspace, size_t ws_bytes, void* stream,
                         pie_fwd_adapter_plan_t** out) {
  using namespace pie;
  if (!out) return set_last_error(PIE_EINVAL, "out is NULL");
  *out = nullptr;
  if (!rank_built(max_rank)) return set_last_error(PIE_EUNSUPPORTED, "max_rank not in {0, 8, 16, 32, 64}");
  if (num_adapters < 0) return set_last_error(PIE_EINVAL, "num_adapters < 0");
  int64_t nt_all = 0;
  int rc = check_lanes(num_lanes, row_indptr, &nt_all);
  if (rc != PIE_OK) return rc;
  if (num_lanes > 0 && !adapter_of_lane) return set_last_error(PIE_EINVAL, "adapter_of_lane is NULL");
  std::vector<ad::Tile> tiles;
  for (int l = 0; l < num_lanes; ++l) {
    const int a = adapter_of_lane[l];
    if (a < -1 || a >= num_adapters)
      return set_last_error(PIE_ERANGE, "adapter id outside [-1, num_adapters)");
    if (a < 0) continue;
    for (int r0 = row_indptr[l]; r0 < row_indptr[l + 1]; r0 += ad::kTileRows)
      tiles.push_back({r0, std::min(ad::kTileRows, row_indptr[l + 1] - r0), a, 0});
  }
  if (tiles.size() > size_t(INT32_MAX)) return set_last_error(PIE_ERANGE, "too many tiles");
  // largest tiles first (the grid's tail is made of the short ones); tiles of
  // one adapter next to each other so that its A and B are read while in L2
  std::stable_sort(tiles.begin(), tiles.end(), [](const ad::Tile& u, const ad::Tile& v) {
    return u.n != v.n ? u.n > v.n : u.adapter < v.adapter;
  });
  const int N = row_indptr[num_lanes];
  const WsLayout Y = ws_layout(nt_all, N, max_rank);
  if (ws_bytes < Y.total || (Y.total > 0 && !dev_workspace))
    return set_last_error(PIE_ENOSPACE, "workspace smaller than pie_fwd_adapter_workspace_bytes()");
  if (reinterpret_cast<uintptr_t>(dev_workspace) % 256 != 0)
    return set_last_error(PIE_EINVAL, "workspace must be 256-byte aligned");

  // the grouped path when every adapter in use serves at most kGMaxRows rows:
  // one group per adapter, its rows in row order
  std::vector<ad::Group> groups;
  std::vector<int32_t> group_rows;
  {
    std::vector<std::vector<int32_t>> by_adapter(size_t(std::max(num_adapters, 0)));
    bool few = true;
    for (int l = 0; l < num_lanes && few; ++l) {
      const int a = adapter_of_lane[l];
      if (a < 0) continue;
      for (int r = row_indptr[l]; r < row_indptr[l + 1]; ++r) by_adapter[size_t(a)].push_back(r);
      few = by_adapter[size_t(a)].size() <= size_t(ad::kGMaxRows);
    }
    if (few) {
      for (int a = 0; a < num_adapters; ++a) {
        std::vector<int32_t>& v = by_adapter[size_t(a)];
        if (v.empty()) continue;
        std::sort(v.begin(), v.end());
        groups.push_back({int32_t(group_rows.size()), int32_t(v.size()), a, 0});
        group_rows.insert(group_rows.end(), v.begin(), v.end());
      }
    }
  }
  // one copy: the tiles, zeroed per-tile counters, the groups and their rows
  const size_t copy = tiles.empty() ? 0 : Y.group_rows + group_rows.size() * 4;
  int err = PIE_OK;
  PinnedBlock* blk = pinned_acquire(std::max<size_t>(copy, 1), &err);
  if (!blk) return err;
  if (copy) {
    std::memset(blk->ptr, 0, copy);
    std::memcpy(blk->ptr, tiles.data(), tiles.size() * sizeof(ad::Tile));
    std::memcpy(static_cast<char*>(blk->ptr) + Y.groups, groups.data(),
                groups.size() * sizeof(ad::Group));
    std::memcpy(static_cast<char*>(blk->ptr) + Y.group_rows, group_rows.data(),
                group_rows.size() * 4);
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (copy && cudaMemcpyAsync(static_cast<char*>(dev_workspace) + Y.tiles, blk->ptr, copy,
                              cudaMemcpyHostToDevice, s) != cudaSuccess) {
    pinned_release(blk);
    return set_last_error(PIE_ECUDA, std::string("adapter plan upload failed: ") +
                                         cudaGetErrorString(cudaGetLastError()));
  }
  if (cudaEventRecord(blk->ev, s) != cudaSuccess)
    return set_last_error(PIE_ECUDA, "cudaEventRecord failed after the adapter plan upload");

  pie_fwd_adapter_plan_t* p = new pie_fwd_adapter_plan_t;
  p->num_lanes = num_lanes;
  p->num_rows = N;
  p->num_adapters = num_adapters;
  p->max_rank = max_rank;
  p->num_tiles = int32_t(tiles.size());
  p->max_tile_rows = 0;
  for (const ad::Tile& t : tiles) p->max_tile_rows = std::max(p->max_tile_rows, t.n);
  p->tiles = reinterpret_cast<ad::Tile*>(static_cast<char*>(dev_workspace) + Y.tiles);
  p->counters = reinterpret_cast<int*>(static_cast<char*>(dev_workspace) + Y.counters);
  p->t_part = reinterpret_cast<float*>(static_cast<char*>(dev_workspace) + Y.t_part);
  p->t_final = reinterpret_cast<float*>(static_cast<char*>(dev_workspace) + Y.t_final);
  p->num_groups = int32_t(groups.size());
  p->max_group_rows = 0;
  for (const ad::Group& gr : groups) p->max_group_rows = std::max(p->max_group_rows, gr.n);
  p->groups = reinterpret_cast<ad::Group*>(static_cast<char*>(dev_workspace) + Y.groups);
  p->group_rows = reinterpret_cast<int32_t*>(static_cast<char*>(dev_workspace) + Y.group_rows);
  p->staging = blk;
  *out = p;
  return PIE_OK;
}

int32_t pie_fwd_adapter_plan_num_tiles(const pie_fwd_adapter_plan_t* plan) {
  return plan ? plan->num_tiles : -1;
}

int32_t pie_fwd_adapter_plan_num_groups(const pie_fwd_adapter_plan_t* plan) {
  return plan ? plan->num_groups : -1;
}

int pie_fwd_adapter_apply(const pie_fwd_adapter_plan_t* plan, int32_t dtype, int32_t d_in,
                          int32_t d_out, int32_t rank, const void* x, void* y, const void* lora_a,
                          const void* lora_b, const float* scale, const void* ia3,
                          uint32_t* status, void* stream) {
  using namespace pie;
  if (!plan) return set_last_error(PIE_EINVAL, "plan is NULL");
  if (dtype != PIE_BF16) return set_last_error(PIE_EUNSUPPORTED, "adapters are built for bf16");
  if (!rank_built(rank)) return set_last_error(PIE_EUNSUPPORTED, "rank not in {0, 8, 16, 32, 64}");
  if (rank > plan->max_rank) return set_last_error(PIE_ERANGE, "rank above the plan's max_rank");
  if (d_in <= 0 || d_in % ad::kChunk != 0)
    return set_last_error(PIE_EUNSUPPORTED, "d_in must be a positive multiple of 64");
  if (d_out <= 0 || d_out % ad::kOBlock != 0)
    return set_last_error(PIE_EUNSUPPORTED, "d_out must be a positive multiple of 256");
  if (plan->num_tiles == 0 || (rank == 0 && !ia3)) return PIE_OK;
  if (!y) return set_last_error(PIE_EINVAL, "y is NULL");
  if (rank > 0 && (!x || !lora_a || !lora_b || !scale))
    return set_last_error(PIE_EINVAL, "x, lora_a, lora_b and scale are required when rank > 0");
  auto misaligned = [](const void* q) { return q && reinterpret_cast<uintptr_t>(q) % 16 != 0; };
  if (misaligned(x) || misaligned(y) || misaligned(lora_a) || misaligned(lora_b))
    return set_last_error(PIE_EINVAL, "x, y, lora_a and lora_b must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(ia3) % 2 != 0)
    return set_last_error(PIE_EINVAL, "ia3 must be 2-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  switch (rank) {
    case 0: e = launch_adapter<0>(*plan, d_in, d_out, x, y, lora_a, lora_b, scale, ia3, status, s); break;
    case 8: e = launch_adapter<8>(*plan, d_in, d_out, x, y, lora_a, lora_b, scale, ia3, status, s); break;
    case 16: e = launch_adapter<16>(*plan, d_in, d_out, x, y, lora_a, lora_b, scale, ia3, status, s); break;
    case 32: e = launch_adapter<32>(*plan, d_in, d_out, x, y, lora_a, lora_b, scale, ia3, status, s); break;
    default: e = launch_adapter<64>(*plan, d_in, d_out, x, y, lora_a, lora_b, scale, ia3, status, s); break;
  }
  if (e != cudaSuccess)
    return set_last_error(PIE_ECUDA, std::string("adapter launch failed: ") + cudaGetErrorString(e));
  return PIE_OK;
}

void pie_fwd_adapter_plan_destroy(pie_fwd_adapter_plan_t* plan) {
  if (!plan) return;
  pie::pinned_release(plan->staging);
  delete plan;
}

}  // extern "C"
