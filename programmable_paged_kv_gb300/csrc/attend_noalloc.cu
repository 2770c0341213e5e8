// Decode attention that allocates nothing.
//
// pie_fwd_decode_attend_noalloc runs the split-KV decode attention and its
// combine step for one query row per lane, taking every input from device
// arrays the caller already owns, and keeps its scratch (work items, combine
// entries and the per-chunk partial softmax states) in one statically sized
// __device__ array of this library instead of a caller workspace.  It exists
// for callers that cannot call cudaMalloc (or any allocator) at the point
// where they launch attention: code that must not allocate device memory
// because it runs under a foreign memory manager with a fixed budget, or a
// host path that may not take the allocator's locks.
//
// The scratch array is shared by every call in the process on a given GPU
// and keeps the previous call's contents.  Nothing in it has to start at
// zero: every call rewrites all the work items, combine entries and partial
// states that it reads.  Calls whose executions overlap on the GPU (on
// different streams, or from different host threads without ordering) race
// on the array and produce wrong outputs; issue them on one stream.
//
// The device address of the array is looked up (cudaGetSymbolAddress) on
// the first call made on each device, with that device current; that first
// call should therefore come before any stream capture on the device.
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>

#include "common.cuh"

namespace pie {

// Maximum scratch: 16 MiB per GPU that loads the library.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
constexpr int kNoAllocChunk = 512;  // slots per split (multiple of kStageSlots)

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

static std::mutex g_noalloc_mu;
static void* g_noalloc_addr[64] = {nullptr};

// Device address of the scratch array on the current device (set-up once
// per device).
static cudaError_t noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return cudaSuccess;
}

// Work items: (lane l, kv head g, chunk c) -> slots [c*CH, min(extent, (c+1)*CH))
// of lane l's single row, where extent = min(kv_len[l], slots[l] + 1) (default
// visibility).  Chunks past the extent are empty items whose partial state is
// (-inf, 0).  extent is clamped to max_kv_len (PIE_STATUS_NOALLOC_TRUNC) and to
// the slots the lane's pages hold (PIE_STATUS_BOUNDS: the page table is device
// data, so it is checked here rather than on the host).
__global__ void noalloc_items_kernel(int L, int Hkv, int MC, int nq, int max_kv_len, int P,
                                     const int32_t* __restrict__ slots,
                                     const int32_t* __restrict__ kv_len,
                                     const int32_t* __restrict__ page_indptr, DecItem* items,
                                     CombEntry* comb, int32_t* readout, uint32_t* status) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < L * Hkv * MC) {
    const int c = i % MC, lg = i / MC, g = lg % Hkv, l = lg / Hkv;
    int ext = min(kv_len[l], slots[l] + 1);
    if (ext > max_kv_len) {
      ext = max_kv_len;
      if (g == 0 && c == 0) set_status(status, PIE_STATUS_NOALLOC_TRUNC);
    }
    const int cap = max(0, page_indptr[l + 1] - page_indptr[l]) * P;
    if (ext > cap) {
      ext = cap;
      if (g == 0 && c == 0) set_status(status, PIE_STATUS_BOUNDS);
    }
    ext = max(ext, 0);
    const int kb = c * kNoAllocChunk;
    const int ke = max(kb, min(ext, kb + kNoAllocChunk));
    items[i] = DecItem{l, g, l, 1, kb, ke, i * nq, -1};  // -1: no compacted list
  }
  if (i < L * Hkv) comb[i] = CombEntry{i * MC * nq, MC, nq, i / Hkv, -1, 0, 0, 0};  // block l = row l
  if (i < L) readout[i] = i;
}

static int nofail(int code, const std::string& m) { return set_last_error(code, m); }

}  // namespace pie

using namespace pie;

extern "C" int pie_fwd_decode_attend_noalloc(const pie_fwd_desc* desc, int32_t num_lanes,
                                             int32_t max_kv_len, const int32_t* slots,
                                             const int32_t* kv_len, const int32_t* page_indptr,
                                             const int32_t* page_ids, int32_t num_pool_pages,
                                             const void* q_rot,
                                             const void* k_pool, const void* v_pool, void* out,
                                             float* lse, uint32_t* status, void* stream) {
  if (!desc) return nofail(PIE_EINVAL, "desc is NULL");
  const pie_fwd_desc& D = *desc;
  if (D.num_q_heads <= 0 || D.num_kv_heads <= 0 || D.num_q_heads % D.num_kv_heads != 0)
    return nofail(PIE_EINVAL, "num_q_heads must be a positive multiple of num_kv_heads");
  if ((D.head_dim != 64 && D.head_dim != 128) ||
      (D.page_size != 8 && D.page_size != 16 && D.page_size != 32) ||
      (D.dtype != PIE_F32 && D.dtype != PIE_BF16))
    return nofail(PIE_EUNSUPPORTED, "head_dim 64/128, page_size 8/16/32, f32/bf16 only");
  const int G = D.num_q_heads / D.num_kv_heads;
  if (G > 8) return nofail(PIE_EUNSUPPORTED, "more than 8 q heads per kv head is not built");
  if (num_lanes < 0 || max_kv_len < 0 || num_pool_pages < 0)
    return nofail(PIE_EINVAL, "negative size");
  if (num_lanes == 0) return PIE_OK;
  if (!slots || !kv_len || !page_indptr || !page_ids || !q_rot || !k_pool || !v_pool || !out)
    return nofail(PIE_EINVAL, "a required pointer is NULL");
  const int L = num_lanes, Hkv = D.num_kv_heads, d = D.head_dim;
  const int nq = G <= 2 ? 2 : (G <= 4 ? 4 : 8);
  const int MC = max_kv_len > 0 ? (max_kv_len + kNoAllocChunk - 1) / kNoAllocChunk : 1;
  const size_t n_items = size_t(L) * Hkv * MC;
  const size_t n_parts = n_items * nq;
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t off_items = 0;
  const size_t off_comb = al(off_items + n_items * sizeof(DecItem));
  const size_t off_ro = al(off_comb + size_t(L) * Hkv * sizeof(CombEntry));
  const size_t off_ml = al(off_ro + size_t(L) * sizeof(int32_t));
  const size_t off_o = al(off_ml + n_parts * sizeof(float2));
  const size_t need = off_o + n_parts * d * sizeof(float);
  if (need > kNoAllocScratchBytes)
    return nofail(PIE_ERANGE, "num_lanes * num_kv_heads * ceil(max_kv_len/512) partial states "
                              "exceed the 16 MiB static scratch of the no-allocation entry point");
  void* base = nullptr;
  cudaError_t e = noalloc_scratch(&base);
  if (e != cudaSuccess)
    return nofail(PIE_ECUDA, std::string("scratch address lookup: ") + cudaGetErrorString(e));
  char* sc = static_cast<char*>(base);

  pie_fwd_plan_t p;
  std::memset(&p, 0, sizeof(p));
  p.device_tables = true;  // the items kernel writes them
  p.desc = D;
  if (p.desc.sm_scale == 0.0f) p.desc.sm_scale = 1.0f / sqrtf(static_cast<float>(d));
  p.L = L;
  p.N = L;
  p.R = L;
  p.G = G;
  p.nq = nq;
  p.num_dec_items = static_cast<int32_t>(n_items);
  p.num_part_slots = static_cast<int64_t>(n_parts);
  p.num_comb_merge = L * Hkv;
  p.dev.slots = slots;
  p.dev.kv_len = kv_len;
  p.dev.page_indptr = page_indptr;
  p.dev.page_ids = page_ids;
  p.dev.num_pool_pages = num_pool_pages;
  p.dev.dec_items = reinterpret_cast<const DecItem*>(sc + off_items);
  p.dev.comb = reinterpret_cast<const CombEntry*>(sc + off_comb);
  p.dev.readout = reinterpret_cast<const int32_t*>(sc + off_ro);
  p.dev.row_block = p.dev.readout;  // one row per lane: row l is block l (identity)
  p.dev.part_ml = reinterpret_cast<float2*>(sc + off_ml);
  p.dev.part_o = reinterpret_cast<float*>(sc + off_o);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int threads = 256;
  const int blocks = static_cast<int>((n_items + threads - 1) / threads);
  noalloc_items_kernel<<<blocks, threads, 0, s>>>(
      L, Hkv, MC, nq, max_kv_len, D.page_size, slots, kv_len, page_indptr,
      reinterpret_cast<DecItem*>(sc + off_items),
      reinterpret_cast<CombEntry*>(sc + off_comb), reinterpret_cast<int32_t*>(sc + off_ro), status);
  e = cudaGetLastError();
  if (e == cudaSuccess) e = launch_attend_decode(p, q_rot, k_pool, v_pool, nullptr, status, s);
  if (e == cudaSuccess) e = launch_combine(p, out, lse, nullptr, nullptr, s);
  if (e != cudaSuccess) return nofail(PIE_ECUDA, std::string("launch: ") + cudaGetErrorString(e));
  return PIE_OK;
}
