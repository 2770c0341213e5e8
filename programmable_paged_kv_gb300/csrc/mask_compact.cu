// Mask pre-pass for masked passes on the list-walking kernels (Pie "The forward
// pass", Attention masks: a row may skip slots it would read under a causal
// mask -- sliding windows, attention sinks, TOVA-style eviction).
//
// Reading only the slots some row can see is what keeps a masked pass near
// its algorithmic bytes: a window of 4,096 slots in a 32,768-slot working set
// touches an eighth of the pages, and a TOVA mask that keeps a quarter of the
// slots touches nearly every page but only a quarter of the slots.  For every
// row block (the rows one tensor-core or split-KV item serves) three small
// kernels build
//   1. the union of the rows' mask words (bits at or past kv_len cleared);
//   2. the compacted list of the slots set in the union, ascending, and its
//      length (and the KV tiles of all blocks' lists, which set how many
//      chunks each block's items split it into);
//   3. each row's mask re-expressed over that list (bit i of a row's word
//      i/32 = the row sees list[i]), and the pool row of every listed slot
//      (its page looked up once here, not by every kv head's item).
// The attention kernels then walk tiles of the list, copying the K/V rows of
// those slots (whole pages when the list is page-granular), and test
// visibility with the re-expressed words exactly as they test plain mask
// words.  The union words are kept in
// the first row of the block's re-expressed mask area until step 3
// overwrites it.

#include "common.cuh"

namespace pie {

// 1. grid (ceil(max_nw / 32), num_blocks), 256 threads: each warp ORs every
// 8th row of the block over 32 consecutive words.
__global__ void __launch_bounds__(256) mask_union_kernel(DevMeta m,
                                                         const uint32_t* mask) {
  __shared__ uint32_t part[8][32];
  grid_dep_wait();    // the kernels before it
  grid_dep_launch();  // the list kernel may start (it waits for this one)
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *m.mask_tiles = 0;
  const MaskBlock B = m.mblocks[blockIdx.y];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int w = blockIdx.x * 32 + lane;
  if (blockIdx.x * 32 >= B.nw) return;
  uint32_t acc = 0;
  if (w < B.nw) {
    // eight of the warp's rows per step, their loads in flight together
    for (int r = B.r0 + warp; r < B.r1; r += 64) {
      uint32_t x[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        x[k] = r + 8 * k < B.r1 ? mask[m.mask_word_indptr[r + 8 * k] + w] : 0u;
#pragma unroll
      for (int k = 0; k < 8; ++k) acc |= x[k];
    }
  }
  part[warp][lane] = acc;
  __syncthreads();
  if (warp == 0 && w < B.nw) {
    uint32_t u = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) u |= part[i][lane];
    const int kv = m.kv_len[B.lane];
    if (w == B.nw - 1 && (kv & 31)) u &= (1u << (kv & 31)) - 1u;
    m.cmask[B.cmask_off + w] = u;
  }
}

// Block-wide sum over the 1024 threads (every thread calls it).
__device__ __forceinline__ int block_sum_1024(int v, int* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  __syncthreads();  // red may still be read from a previous call
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = lane < 32 ? red[lane] : 0;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Pages (P-bit groups) of a union word with at least one set slot.
__device__ __forceinline__ int pages_set(uint32_t u, int P) {
  int n = 0;
  for (int g = 0; g < 32; g += P) n += ((u >> g) & ((P == 32) ? 0xFFFFFFFFu : ((1u << P) - 1u))) != 0;
  return n;
}

// 2. one CTA of 1024 threads per block: the list of the block's visible
// slots and its length.  When the pages holding a visible slot add at most a
// quarter to the visible slots (a window: long runs), the list is
// page-granular -- every slot below kv_len of each such page, in page order,
// so the tensor-core kernel can load whole pages with one box copy each;
// otherwise (scattered slots, e.g. TOVA) it lists only the visible slots,
// which the kernel gathers row by row.  Both are ascending.
__global__ void __launch_bounds__(1024) mask_list_kernel(DevMeta m, int P, int BN) {
  __shared__ int warp_tot[32];
  __shared__ int red[32];
  __shared__ int chunk_total;
  grid_dep_wait();  // the union kernel's words
  grid_dep_launch();
  const int b = blockIdx.x;
  const MaskBlock B = m.mblocks[b];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kv = m.kv_len[B.lane];
  // pass 1: visible slots and pages with a visible slot
  int cs = 0, cp = 0;
  for (int w = threadIdx.x; w < B.nw; w += 1024) {
    const uint32_t u = m.cmask[B.cmask_off + w];
    cs += __popc(u);
    cp += pages_set(u, P);
  }
  const int n_slots = block_sum_1024(cs, red);
  const int n_pages = block_sum_1024(cp, red);
  const bool page_mode = n_slots > 0 && int64_t(n_pages) * P * 4 <= int64_t(n_slots) * 5;
  int32_t* list = m.list + B.list_off;
  // pass 2: exclusive prefix over words of the entries each word contributes
  int running = 0;
  for (int base = 0; base < B.nw; base += 1024) {
    const int w = base + threadIdx.x;
    const uint32_t u = w < B.nw ? m.cmask[B.cmask_off + w] : 0u;
    const int c = page_mode ? pages_set(u, P) : __popc(u);
    int incl = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int t = warp_tot[lane];
      int ti = t;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, ti, off);
        if (lane >= off) ti += v;
      }
      warp_tot[lane] = ti - t;  // exclusive prefix over warps
      if (lane == 31) chunk_total = ti;
    }
    __syncthreads();
    const int pos = running + warp_tot[warp] + incl - c;
    if (page_mode) {
      // the word's pages with a visible slot: all of their slots below kv_len
      int k = 0;
      for (int g = 0; g < 32; g += P) {
        const uint32_t grp = (u >> g) & ((P == 32) ? 0xFFFFFFFFu : ((1u << P) - 1u));
        if (grp == 0u) continue;
        const int s0 = w * 32 + g;
        for (int off = 0; off < P && s0 + off < kv; ++off) list[(pos + k) * P + off] = s0 + off;
        ++k;
      }
    } else {
      // the warp writes its 32 words' entries one word at a time: lane i
      // stores bit i of the word at its rank, so every store is coalesced
      const uint32_t below = (1u << lane) - 1u;
      for (int k = 0; k < 32; ++k) {
        const uint32_t uk = __shfl_sync(0xffffffffu, u, k);
        if (uk == 0u) continue;  // uniform across the warp
        const int pk = __shfl_sync(0xffffffffu, pos, k);
        const int wk = __shfl_sync(0xffffffffu, w, k);
        if ((uk >> lane) & 1u) list[pk + __popc(uk & below)] = wk * 32 + lane;
      }
    }
    running += chunk_total;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    // page mode: the last listed page is cut at kv_len when it is the lane's
    // last, partly filled page (its slots at/after kv_len are never listed)
    int len = page_mode ? running * P : running;
    if (page_mode && (kv % P) != 0) {
      const int last_page = (kv - 1) / P;
      const uint32_t u = m.cmask[B.cmask_off + (last_page * P) / 32];
      const int g = (last_page * P) % 32;
      if (((u >> g) & ((P == 32) ? 0xFFFFFFFFu : ((1u << P) - 1u))) != 0u) len -= P - (kv % P);
    }
    m.list_len[b] = len;
    m.list_mode[b] = page_mode ? 1 : 0;
    atomicAdd(m.mask_tiles, (len + BN - 1) / BN);  // KV tiles of all blocks' lists
  }
}

// 3. grid (ceil(max_nw / 8), num_blocks, row groups), 256 threads: warp ->
// one word of list positions and 16 rows of the block; for each row, ballot
// the row's bit at each of the 32 listed slots (all 16 rows' loads in flight
// together).  The first row group's threads also write their listed slots'
// pool rows.
__global__ void __launch_bounds__(256) mask_cmask_kernel(DevMeta m,
                                                         const uint32_t* mask,
                                                         int Hkv, int P) {
  grid_dep_wait();  // the list kernel's lists
  grid_dep_launch();
  const int b = blockIdx.y;
  const MaskBlock B = m.mblocks[b];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cw = blockIdx.x * 8 + warp;
  const int U = m.list_len[b];
  if (cw >= B.nw || cw * 32 >= U) return;
  const int i = cw * 32 + lane;
  const int r0 = B.r0 + 16 * blockIdx.z;
  if (r0 >= B.r1) return;
  const int slot = i < U ? m.list[B.list_off + i] : -1;
  if (slot >= 0 && blockIdx.z == 0)
    m.lrow[B.list_off + i] = m.page_ids[m.page_indptr[B.lane] + slot / P] * Hkv * P + slot % P;
  uint32_t w[16];
#pragma unroll
  for (int k = 0; k < 16; ++k)
    w[k] = (slot >= 0 && r0 + k < B.r1) ? mask[m.mask_word_indptr[r0 + k] + (slot >> 5)] : 0u;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const uint32_t bal = __ballot_sync(0xffffffffu, ((w[k] >> (slot & 31)) & 1u) != 0);
    if (lane == 0 && r0 + k < B.r1) m.cmask[B.cmask_off + int64_t(r0 + k - B.r0) * B.nw + cw] = bal;
  }
}

cudaError_t launch_mask_compact(const pie_fwd_plan_t& p, const uint32_t* mask_words,
                                cudaStream_t s) {
  const int nb = p.num_mblocks, nw = p.mblock_max_nw;
  if (nb == 0 || nw == 0) return cudaSuccess;
  cudaError_t e = launch_dependent(mask_union_kernel, dim3((nw + 31) / 32, nb), dim3(256), 0, s,
                                   true, p.dev, mask_words);
  if (e != cudaSuccess) return e;
  e = launch_dependent(mask_list_kernel, dim3(nb), dim3(1024), 0, s, true, p.dev,
                       p.desc.page_size, tc_kv_tile(p.tc_nt));
  if (e != cudaSuccess) return e;
  const int row_groups = (p.mblock_max_rows + 15) / 16;
  return launch_dependent(mask_cmask_kernel, dim3((nw + 7) / 8, nb, row_groups), dim3(256), 0, s,
                          true, p.dev, mask_words, p.desc.num_kv_heads, p.desc.page_size);
}

}  // namespace pie
